"""CPU fp64 oracle for KV-cache attention: GQA/MHA/MQA decode, causal GQA prefill,
MLA (absorbed and decompressed), the log-sum-exp merge of split partials, the rotary
embedding and cache append of a decode step, decode over an fp8 (E4M3) cache, chunked
prefill over an existing cache (GQA and MLA), and the KV-cache byte/parameter accounting
the pages print.

This package is TEST INFRASTRUCTURE. It is the plain, slow definition that the CUDA
library is checked against. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The product path (the C-ABI library and
its Python binding) never imports, calls or links anything here, and nothing here
imports the product path: the two share no code. Inputs are plain NumPy arrays (any
float dtype); all arithmetic is float64.

Sources (cited by page title and section):
  * "模型架构｜MQA & GQA 调研" (lichtung612 blog): definitions of MHA/MQA/GQA-G (section
    "Grouped-query attention"), the ``repeat_kv`` helper and ``Attention.forward``
    (section "代码"): scores = q·kᵀ/√d, + mask, softmax in fp32, · v, over a cache that
    already holds the new token.
  * "MHA, MQA và GQA" (coregenaihub interactive ebook): byte/parameter table for the
    Llama-3-8B shape and the rule that the KV-group count must divide the Q-head count.
  * "Attention Architecture Experiments" (minimind docs), section "Benchmark": KV floats
    per token per layer, GQA 2·4·96 = 768 vs MLA 128 + 48 = 176.
  * qqstock article on DeepSeek MLA, sections 1-3 and 6 and its
    ``MultiHeadLatentAttention`` code: low-rank joint KV compression, weight absorption,
    decoupled RoPE key shared by all heads, and "V shares the activation with the
    un-RoPE'd K".

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (brute
force, closed forms, a library cross-check, identities and the pages' printed values);
none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    check_grouping,
    kv_head_for_query_head,
    repeat_kv,
    attend,
    attend_partial,
    lse_merge,
    decode_gqa,
    decode_gqa_unit,
    prefill_gqa_causal,
)
from .mla import (  # noqa: F401
    absorb_query,
    apply_uv,
    mla_decode_absorbed,
    mla_decode_naive,
)
from .rope import (  # noqa: F401
    rope_rotate,
    kv_append_rope,
    mla_append_rope,
)
from .fp8 import (  # noqa: F401
    e4m3_to_float,
    dequantize,
    decode_gqa_fp8,
)
from .chunked import (  # noqa: F401
    prefill_gqa_chunked,
    mla_prefill_absorbed,
    mla_prefill_naive,
)
from . import accounting  # noqa: F401
