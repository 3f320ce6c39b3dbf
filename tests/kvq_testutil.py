"""Shared helpers of the GPU tests: build a device cache and an oracle cache
from the same host arrays, and compare their bytes and outputs."""

import numpy as np
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_08_gb300 import build as kbuild
from quantized_kv_cache_08_gb300.cache import KVCache

ATOL = 2e-3   # max abs error of attention outputs against the fp64 oracle


def need_gpu():
    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA GPU; the library has no CPU fallback")
    kbuild.build()


def to_dev(x):
    return x.contiguous().cuda()


def oracle_input(x):
    """Exact float64 view of a float32/bfloat16 host tensor."""
    return x.float().numpy().astype(np.float64)


def assert_rows_equal(cache, oracle, seq, lo, hi):
    """Device bytes of logical rows [lo, hi) equal the oracle's bytes."""
    plo, phi = cache.physical_rows(seq, lo, hi)
    kd = cache.k_rows(seq, plo, phi).cpu().numpy()
    vd = cache.v_rows(seq, plo, phi).cpu().numpy()
    ko, vo = oracle.rows(seq, lo, hi)
    if not np.array_equal(kd, ko):
        bad = np.argwhere(kd != ko)
        raise AssertionError(f"K bytes differ in seq {seq} at {len(bad)} places, first {bad[:5].tolist()}")
    if not np.array_equal(vd, vo):
        bad = np.argwhere(vd != vo)
        raise AssertionError(f"V bytes differ in seq {seq} at {len(bad)} places, first {bad[:5].tolist()}")


def assert_close(got, want, atol=ATOL, what="output"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    mask = ~np.isnan(want)
    assert np.all(np.isfinite(got[mask])), f"{what}: non-finite values"
    err = np.max(np.abs(got[mask] - want[mask])) if mask.any() else 0.0
    assert err <= atol, f"{what}: max abs error {err:.3e} > {atol:.1e}"
    return err


class Pair:
    """A device cache and an oracle cache fed with identical inputs."""

    def __init__(self, n_seq, n_kv, head_dim, n_q, max_t=1, max_rows=0, window=0, ring=False,
                 fmt="q8_0/q5_1"):
        self.dev = KVCache(n_seq, n_kv, head_dim, n_q, max_t=max_t, max_rows=max_rows,
                           window=window, ring=ring, fmt=fmt)
        self.ora = O.OracleKvCache(n_seq, n_kv, head_dim, window=window, fmt=fmt)
        self.n_seq, self.n_kv, self.head_dim, self.n_q = n_seq, n_kv, head_dim, n_q

    def append(self, k, v, seq_ids=None):
        """k, v: host float32/bf16 [n, T, n_kv, head_dim]."""
        self.dev.append(to_dev(k), to_dev(v), seq_ids=seq_ids)
        self.ora.append(k.float().numpy(), v.float().numpy(), seq_ids=seq_ids)

    def decode(self, q, sinks=None, scale=0.0, **okw):
        out = self.dev.decode(to_dev(q), sinks=None if sinks is None else to_dev(sinks), scale=scale)
        ref = self.ora.decode(oracle_input(q), sinks=None if sinks is None else sinks.double().numpy(),
                              scale=None if scale <= 0 else scale, **okw)
        return out.cpu().numpy(), ref

    def truncate(self, new_len):
        self.dev.truncate(new_len)
        self.ora.truncate(new_len)
