"""A torch-facing holder for one kvq layer cache.

PyTorch only provides the device memory (uint8 / int32 tensors) and the
stream; every operation is one call through the C ABI (see _binding).
"""

from __future__ import annotations

import torch

from . import _binding as B


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t):
    if t.dtype == torch.float32:
        return B.KVQ_F32
    if t.dtype == torch.bfloat16:
        return B.KVQ_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _check_dev(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class KVCache:
    """n_seq sequences of one attention layer: q8_0 K plane and q5_1 V plane
    (fmt "q8_0/q5_1") or FP8 E4M3 K and V planes (fmt "e4m3"), device counters
    and the decode workspace, all caller-owned torch memory."""

    FORMATS = {"q8_0/q5_1": (B.KVQ_Q8_0, B.KVQ_Q5_1, 34, 24), "e4m3": (B.KVQ_FP8_E4M3, B.KVQ_FP8_E4M3, 32, 32)}

    def __init__(self, n_seq, n_kv_heads, head_dim, max_q_heads, max_t=1, max_rows=0,
                 window=0, ring=False, device=None, stream=None, fmt="q8_0/q5_1"):
        if fmt not in self.FORMATS:
            raise ValueError(f"fmt must be one of {sorted(self.FORMATS)}")
        k_fmt, v_fmt, _, _ = self.FORMATS[fmt]
        self.fmt = fmt
        self.cfg = B.make_config(n_seq, n_kv_heads, head_dim, max_q_heads, max_t, max_rows,
                                 window, ring, k_fmt, v_fmt)
        sz = B.kvq_required_bytes(self.cfg)
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.k_plane = torch.empty(sz.k_plane, dtype=torch.uint8, device=dev)
        self.v_plane = torch.empty(sz.v_plane, dtype=torch.uint8, device=dev)
        self.counters = torch.empty(sz.counters // 4, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(max(sz.workspace, 16), dtype=torch.uint8, device=dev)
        self.n_seq, self.n_kv_heads, self.head_dim = n_seq, n_kv_heads, head_dim
        # the geometry as the library lays it out
        self.k_tok, self.v_tok, self.rows = sz.k_row_bytes, sz.v_row_bytes, sz.rows
        self.window, self.ring = window, bool(ring)
        self.handle = B.kvq_alloc(self.cfg, self.k_plane.data_ptr(), self.v_plane.data_ptr(),
                                  self.counters.data_ptr(), self.workspace.data_ptr(),
                                  _stream_handle(stream))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None:
            B.kvq_free(h)
            self.handle = None

    # -- the calls of the path: append, decode, truncate (host or device counts)
    def append(self, k, v, seq_ids=None, stream=None):
        """k, v: [n, T, Hkv, D] float32/bfloat16 CUDA tensors."""
        _check_dev(k, "k")
        _check_dev(v, "v")
        if k.shape != v.shape or k.dtype != v.dtype or k.dim() != 4:
            raise ValueError("k and v must both be [n, T, Hkv, D] of one dtype")
        n = self.n_seq if seq_ids is None else len(seq_ids)
        if k.shape[0] != n or k.shape[2] != self.n_kv_heads or k.shape[3] != self.head_dim:
            raise ValueError(f"k shape {tuple(k.shape)} does not match the cache")
        B.kvq_append(self.handle, k.data_ptr(), v.data_ptr(), _dtype_code(k), k.shape[1],
                     seq_ids, _stream_handle(stream))

    def decode(self, q, sinks=None, scale=0.0, out=None, stream=None):
        """q: [n_seq, T, Hq, D] float32/bfloat16; returns float32 [n_seq, T, Hq, D]."""
        _check_dev(q, "q")
        if q.dim() != 4 or q.shape[0] != self.n_seq or q.shape[3] != self.head_dim:
            raise ValueError(f"q shape {tuple(q.shape)} does not match the cache")
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _check_dev(out, "out")
        if out.dtype != torch.float32 or out.shape != q.shape:
            raise ValueError("out must be float32 with q's shape")
        sp = None
        if sinks is not None:
            _check_dev(sinks, "sinks")
            if sinks.dtype != torch.float32 or sinks.numel() != q.shape[2]:
                raise ValueError("sinks must be float32 [Hq]")
            sp = sinks.data_ptr()
        B.kvq_decode(self.handle, q.data_ptr(), _dtype_code(q), q.shape[1], q.shape[2], sp,
                     scale, out.data_ptr(), _stream_handle(stream))
        return out

    def truncate(self, new_len, stream=None):
        B.kvq_truncate(self.handle, list(new_len), _stream_handle(stream))

    def truncate_device(self, accept, T, stream=None):
        """Keep the first accept[b] of each sequence's last T rows; accept is a
        CUDA int32 tensor [n_seq] read when the kernel runs (no host wait)."""
        _check_dev(accept, "accept")
        if accept.dtype != torch.int32 or accept.numel() != self.n_seq:
            raise ValueError("accept must be int32 [n_seq]")
        B.kvq_truncate_device(self.handle, accept.data_ptr(), T, _stream_handle(stream))

    def sync_len(self, stream=None):
        """Wait for the stream and read the device lengths into the host mirror."""
        B.kvq_sync_len(self.handle, _stream_handle(stream))

    # -- host-side helpers
    def lens(self):
        return B.kvq_get_len(self.handle, self.n_seq)[0]

    def bases(self):
        return B.kvq_get_len(self.handle, self.n_seq)[1]

    def note_replayed(self, steps, T):
        B.kvq_note_replayed(self.handle, steps, T)

    def ring_headroom(self, T):
        return B.kvq_ring_headroom(self.handle, T)

    def physical_rows(self, seq, start, end):
        return B.kvq_physical_rows(self.handle, seq, start, end)

    def device_error(self, stream=None):
        return B.kvq_read_device_error(self.handle, _stream_handle(stream))

    def set_split_rows(self, rows):
        B.kvq_set_split_rows(self.handle, rows)

    def set_row_slices(self, slices):
        """Row slices per tile on the stream-K kernel: 0 automatic, 1 or 2."""
        B.kvq_set_row_slices(self.handle, slices)

    def set_softcap(self, softcap):
        """softcap > 0 caps scaled scores to softcap * tanh(s / softcap); 0 is off."""
        B.kvq_set_softcap(self.handle, softcap)

    def set_decode_path(self, path, query_bits=0):
        """path: 0 auto, 1 generic split kernel, 2 stream-K kernel."""
        B.kvq_set_decode_path(self.handle, path, query_bits)

    def k_rows(self, seq, phys_lo, phys_hi):
        """Raw K bytes of physical rows [phys_lo, phys_hi) of a sequence (a view)."""
        n = self.n_seq * self.rows * self.k_tok
        v = self.k_plane[:n].view(self.n_seq, self.rows, self.k_tok)
        return v[seq, phys_lo:phys_hi]

    def v_rows(self, seq, phys_lo, phys_hi):
        n = self.n_seq * self.rows * self.v_tok
        v = self.v_plane[:n].view(self.n_seq, self.rows, self.v_tok)
        return v[seq, phys_lo:phys_hi]
