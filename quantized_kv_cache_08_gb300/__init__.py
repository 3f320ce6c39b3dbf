"""GB300-native quantised KV cache: q8_0 K / q5_1 V (or FP8 E4M3 K and V)
append, truncate (with host or device-held accepted counts) and split-K
flash-decode attention, behind a C ABI (include/kvq.h) implemented by
hand-written sm_103a CUDA kernels in libkvq.so.

`_binding` mirrors the C calls one to one (ctypes); `cache.KVCache` holds the
torch-allocated device buffers of one layer cache; `inputs` draws the seeded
synthetic workloads; `build.build()` compiles the library.
"""

from ._binding import (  # noqa: F401
    EXPORTS, KVQ_BF16, KVQ_F32, KVQ_FP8_E4M3, KVQ_Q5_1, KVQ_Q8_0, KvqError, kvq_alloc, kvq_append,
    kvq_block_bytes, kvq_bytes_per_token, kvq_decode, kvq_decode_noalloc, kvq_free, kvq_get_len, kvq_last_error,
    kvq_note_replayed, kvq_physical_rows, kvq_read_device_error, kvq_required_bytes,
    kvq_ring_headroom, kvq_set_decode_path, kvq_set_softcap, kvq_set_split_rows, kvq_sync_len, kvq_truncate,
    kvq_truncate_device, lib,
    make_config,
)
