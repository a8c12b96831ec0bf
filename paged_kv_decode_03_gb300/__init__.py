"""GB300-native paged-KV decode attention.

Python face of the C-ABI library ``libpagedkv.so`` (declared in
``include/pagedkv.h``): ``paged_kv_append`` and ``paged_decode_attention``,
plus the two steps of the split-KV path (``paged_decode_split_partial``,
``paged_decode_lse_combine``) and a whole model step over one layout
(``paged_decode_step``), chunk attention (``paged_prefill_attention``) and
RoPE fused with the append (``paged_rope_cos_sin_table``,
``paged_kv_append_rope``).  The binding only marshals arguments; every
step of the computation runs in the library's sm_103a kernels.  There is no
CPU fallback: if the library is missing, the first call raises.
"""
from .binding import (  # noqa: F401
    PKV_BF16, PKV_INT8, SCALE_NONE, SCALE_PER_TOKEN, SCALE_PER_HEAD, SPLIT_AUTO, OUT_BF16, OUT_F32,
    PagedKVPool, paged_kv_append, paged_kv_slot_mapping, paged_decode_attention, paged_decode_split_partial,
    paged_decode_lse_combine, paged_decode_workspace_bytes, paged_decode_num_splits,
    paged_decode_split_tokens, PagedKVError, paged_decode_attention_noalloc,
    paged_decode_partial_workspace_bytes, uses_tensor_cores, last_launch_count,
    STATIC_SCRATCH_BYTES, DecodeLayer, paged_prefill_attention, check_bounded_wait, paged_decode_step, paged_decode_step_workspace_bytes,
    library_path, load_library, device_status, exported_symbols,
    ROPE_HALVES, ROPE_INTERLEAVED, paged_rope_cos_sin_table, paged_kv_append_rope,
)
