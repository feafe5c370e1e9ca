"""Plain, slow CPU oracle for paged-KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may use it.  It shares no code with the CUDA
library (``paged_kv_cache_52_gb300``) and imports nothing from it.

Everything is numpy in float64.  bf16 tensors are handled as their raw 16-bit
patterns (``numpy.uint16``) and widened exactly to float64 where arithmetic
starts.  See ``oracle.paged_attention`` for the functions and the passages of
the pages that each one follows.
"""

from .paged_attention import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    kv_append,
    kv_append_checked,
    gather_sequence_kv,
    attention,
    paged_decode_attention,
    paged_prefill_attention,
    online_softmax_attention,
    split_partials,
    merge_partials,
    kv_bytes_per_token_per_layer,
    kv_bytes_per_token,
    kv_cache_bytes,
)

from .fp8_cache import (  # noqa: F401,E402
    e4m3_bits_to_f64,
    f32_to_e4m3_bits,
    quantize_rows,
    kv_append_fp8,
    dequantize,
    paged_decode_attention_fp8,
    paged_prefill_attention_fp8,
)

from .block_manager import (  # noqa: F401,E402
    BlockManager,
    NoFreeBlocks,
    fnv1a64,
    block_hash,
    copy_blocks,
    num_blocks_for_budget,
)
