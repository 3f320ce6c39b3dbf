"""ctypes binding of the kvq C ABI (include/kvq.h), same names as the C calls.

Argument marshalling only: every step of append, decode and truncate runs in
the CUDA kernels of libkvq.so.  Pointer arguments are integers (device
addresses, e.g. ``tensor.data_ptr()``) and streams are ``cudaStream_t`` values
(e.g. ``torch.cuda.current_stream().cuda_stream``) or 0.  A missing library is
an error: there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_ERANGE, KVQ_ECUDA, KVQ_EUNSUPPORTED = 0, 1, 2, 3, 4
KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20
KVQ_F32, KVQ_BF16 = 0, 1
KVQ_Q8_0, KVQ_Q5_1, KVQ_FP8_E4M3 = 0, 1, 2

STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_EINVAL", 2: "KVQ_ERANGE", 3: "KVQ_ECUDA", 4: "KVQ_EUNSUPPORTED"}

# every symbol include/kvq.h declares
EXPORTS = (
    "kvq_required_bytes", "kvq_alloc", "kvq_free", "kvq_append", "kvq_decode",
    "kvq_decode_noalloc", "kvq_truncate", "kvq_truncate_device", "kvq_sync_len", "kvq_get_len", "kvq_note_replayed", "kvq_ring_headroom",
    "kvq_physical_rows", "kvq_read_device_error", "kvq_set_split_rows", "kvq_set_row_slices", "kvq_set_decode_path",
    "kvq_set_softcap",
    "kvq_block_bytes", "kvq_bytes_per_token", "kvq_last_error",
)


class KvqError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class kvq_config(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("max_q_heads", ctypes.c_int), ("max_t", ctypes.c_int), ("max_rows", ctypes.c_int),
        ("window", ctypes.c_int), ("ring", ctypes.c_int), ("k_fmt", ctypes.c_int),
        ("v_fmt", ctypes.c_int),
    ]


class kvq_sizes(ctypes.Structure):
    _fields_ = [("k_plane", ctypes.c_size_t), ("v_plane", ctypes.c_size_t),
                ("counters", ctypes.c_size_t), ("workspace", ctypes.c_size_t),
                ("rows", ctypes.c_int), ("k_row_bytes", ctypes.c_int), ("v_row_bytes", ctypes.c_int)]


_LIB = None


def lib():
    """Load libkvq.so (build it first with quantized_kv_cache_08_gb300.build)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -m quantized_kv_cache_08_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        IP = ctypes.POINTER(ctypes.c_int)
        sig = {
            "kvq_required_bytes": (I, [ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_sizes)]),
            "kvq_alloc": (I, [ctypes.POINTER(kvq_config), P, P, P, P, P, ctypes.POINTER(P)]),
            "kvq_free": (None, [P]),
            "kvq_append": (I, [P, P, P, I, I, IP, I, P]),
            "kvq_decode": (I, [P, P, I, I, I, P, ctypes.c_float, P, P]),
            "kvq_decode_noalloc": (I, [P, P, I, I, I, P, ctypes.c_float, P, P]),
            "kvq_truncate": (I, [P, IP, P]),
            "kvq_truncate_device": (I, [P, P, I, P]),
            "kvq_sync_len": (I, [P, P]),
            "kvq_get_len": (I, [P, IP, IP]),
            "kvq_note_replayed": (I, [P, I, I]),
            "kvq_ring_headroom": (I, [P, I, IP]),
            "kvq_physical_rows": (I, [P, I, I, I, IP, IP]),
            "kvq_read_device_error": (I, [P, IP, P]),
            "kvq_set_split_rows": (I, [P, I]),
            "kvq_set_row_slices": (I, [P, I]),
            "kvq_set_decode_path": (I, [P, I, I]),
            "kvq_set_softcap": (I, [P, ctypes.c_float]),
            "kvq_block_bytes": (I, [I]),
            "kvq_bytes_per_token": (S, [ctypes.POINTER(kvq_config)]),
            "kvq_last_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status):
    if status != KVQ_OK:
        raise KvqError(status, lib().kvq_last_error().decode())


def _ints(xs):
    arr = (ctypes.c_int * len(xs))(*[int(x) for x in xs])
    return arr


def make_config(n_seq, n_kv_heads, head_dim, max_q_heads, max_t=1, max_rows=0, window=0, ring=0,
                k_fmt=KVQ_Q8_0, v_fmt=KVQ_Q5_1):
    return kvq_config(n_seq, n_kv_heads, head_dim, max_q_heads, max_t, max_rows, window,
                      int(bool(ring)), k_fmt, v_fmt)


def kvq_required_bytes(cfg):
    out = kvq_sizes()
    _check(lib().kvq_required_bytes(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def kvq_alloc(cfg, k_plane, v_plane, counters, workspace, stream=0):
    h = ctypes.c_void_p()
    _check(lib().kvq_alloc(ctypes.byref(cfg), k_plane, v_plane, counters, workspace, stream,
                           ctypes.byref(h)))
    return h


def kvq_free(handle):
    lib().kvq_free(handle)


def kvq_append(handle, k, v, dtype, T, seq_ids=None, stream=0):
    if seq_ids is None:
        _check(lib().kvq_append(handle, k, v, dtype, T, None, 0, stream))
    else:
        arr = _ints(seq_ids)
        _check(lib().kvq_append(handle, k, v, dtype, T, arr, len(seq_ids), stream))


def kvq_decode(handle, q, dtype, T, n_q_heads, sinks, scale, out, stream=0):
    _check(lib().kvq_decode(handle, q, dtype, T, n_q_heads, sinks, float(scale), out, stream))


def kvq_decode_noalloc(handle, q, dtype, T, n_q_heads, sinks, scale, out, stream=0):
    _check(lib().kvq_decode_noalloc(handle, q, dtype, T, n_q_heads, sinks, float(scale), out, stream))


def kvq_truncate(handle, new_len, stream=0):
    _check(lib().kvq_truncate(handle, _ints(new_len), stream))


def kvq_truncate_device(handle, accept_d, T, stream=0):
    _check(lib().kvq_truncate_device(handle, accept_d, T, stream))


def kvq_sync_len(handle, stream=0):
    _check(lib().kvq_sync_len(handle, stream))


def kvq_get_len(handle, n_seq):
    lens = (ctypes.c_int * n_seq)()
    bases = (ctypes.c_int * n_seq)()
    _check(lib().kvq_get_len(handle, lens, bases))
    return list(lens), list(bases)


def kvq_note_replayed(handle, steps, T):
    _check(lib().kvq_note_replayed(handle, steps, T))


def kvq_ring_headroom(handle, T):
    n = ctypes.c_int()
    _check(lib().kvq_ring_headroom(handle, T, ctypes.byref(n)))
    return n.value


def kvq_physical_rows(handle, seq, start, end):
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(lib().kvq_physical_rows(handle, seq, start, end, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def kvq_read_device_error(handle, stream=0):
    e = ctypes.c_int()
    _check(lib().kvq_read_device_error(handle, ctypes.byref(e), stream))
    return e.value


def kvq_set_split_rows(handle, rows):
    _check(lib().kvq_set_split_rows(handle, rows))


def kvq_set_row_slices(handle, slices):
    _check(lib().kvq_set_row_slices(handle, slices))


def kvq_set_decode_path(handle, path, query_bits=0):
    _check(lib().kvq_set_decode_path(handle, path, query_bits))


def kvq_set_softcap(handle, softcap):
    _check(lib().kvq_set_softcap(handle, float(softcap)))


def kvq_block_bytes(fmt):
    return lib().kvq_block_bytes(fmt)


def kvq_bytes_per_token(cfg):
    return lib().kvq_bytes_per_token(ctypes.byref(cfg))


def kvq_last_error():
    return lib().kvq_last_error().decode()
