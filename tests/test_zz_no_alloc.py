"""kvq_decode_noalloc: the decode through the library's fixed device scratch
gives the same bytes as kvq_decode through the cache's workspace, call after
call, and refuses a decode whose partials would not fit.

The file name sorts last so the tests also run after every other test in the
same process (the scratch array is shared by all calls on a device)."""

import pytest
import torch

from quantized_kv_cache_08_gb300 import _binding as B
from quantized_kv_cache_08_gb300.cache import KVCache, _dtype_code
from tests.kvq_testutil import need_gpu

pytestmark = pytest.mark.gpu


def _need_gpu():
    need_gpu()      # raises without a GPU: there is no CPU fallback to test


def _noalloc(cache, q, sinks=None, scale=0.0):
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    B.kvq_decode_noalloc(cache.handle, q.data_ptr(), _dtype_code(q), q.shape[1], q.shape[2],
                         None if sinks is None else sinks.data_ptr(), scale, out.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    return out


def _filled(n_seq, Hkv, D, Hq, lens, seed, **kw):
    g = torch.Generator().manual_seed(seed)
    c = KVCache(n_seq, Hkv, D, Hq, max_t=64, max_rows=max(lens) + 8, **kw)
    for b, L in enumerate(lens):
        k = torch.randn(1, L, Hkv, D, generator=g).cuda()
        v = torch.randn(1, L, Hkv, D, generator=g).cuda()
        for t0 in range(0, L, 64):
            c.append(k[:, t0:t0 + 64], v[:, t0:t0 + 64], seq_ids=[b])
    return c, g


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("shape", [
    # n_seq, Hkv, D, Hq, lens, T, sinks, q dtype
    (1, 8, 128, 32, [4096], 1, False, torch.bfloat16),
    (3, 2, 128, 8, [700, 1, 333], 1, True, torch.float32),
    (1, 4, 256, 16, [900], 8, True, torch.float32),
])
def test_noalloc_matches_decode_two_calls(shape, path):
    _need_gpu()
    n_seq, Hkv, D, Hq, lens, T, use_sinks, qdt = shape
    c, g = _filled(n_seq, Hkv, D, Hq, lens, seed=11)
    c.set_decode_path(path)
    q = torch.randn(n_seq, T, Hq, D, generator=g).to(qdt).cuda()
    sinks = torch.randn(Hq, generator=g).cuda() if use_sinks else None
    ref = c.decode(q, sinks=sinks)
    first = _noalloc(c, q, sinks)
    second = _noalloc(c, q, sinks)
    torch.cuda.synchronize()
    assert torch.equal(first, ref)
    assert torch.equal(second, ref)
    # and the workspace entry point is unaffected by the no-alloc calls
    assert torch.equal(c.decode(q, sinks=sinks), ref)
    assert c.device_error() == 0


def test_noalloc_refuses_oversize_partials():
    _need_gpu()
    # 64-row splits over 32768 rows: 512 splits x 64 queries x (128 + 2)
    # floats is about 17 MB, above the 16 MiB scratch
    c = KVCache(1, 8, 128, 64, max_t=1, max_rows=32768)
    c.set_decode_path(1)
    c.set_split_rows(64)
    k = torch.randn(1, 1, 8, 128, device="cuda")
    c.append(k, k)
    q = torch.randn(1, 1, 64, 128, device="cuda")
    with pytest.raises(B.KvqError) as e:
        _noalloc(c, q)
    assert e.value.status == B.KVQ_ERANGE
    assert "no-alloc" in str(e.value)
    # the workspace entry point still serves the same decode
    out = c.decode(q)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("name", ["ctx512", "ctx32k", "batch64", "swa_ring", "spec_verify"])
def test_noalloc_fits_every_workload_at_full_size(name):
    """Each of the five decode workloads at its full size (automatic kernel
    choice, as benchmarked) fits the 16 MiB scratch, and the no-alloc decode
    gives the bytes of the workspace decode."""
    _need_gpu()
    from quantized_kv_cache_08_gb300.inputs import workload
    wl = workload(name)
    lens = [2 * wl.window] if wl.ring else list(wl.lengths())
    c = KVCache(wl.n_seq, wl.n_kv, wl.head_dim, wl.n_q, max_t=512,
                max_rows=0 if wl.ring else max(lens) + wl.T, window=wl.window, ring=wl.ring)
    g = torch.Generator(device="cuda").manual_seed(5)
    for b, L in enumerate(lens):
        for t0 in range(0, L, 512):
            n = min(512, L - t0)
            k = torch.randn(1, n, wl.n_kv, wl.head_dim, generator=g, device="cuda")
            v = torch.randn(1, n, wl.n_kv, wl.head_dim, generator=g, device="cuda")
            c.append(k, v, seq_ids=[b])
    q = torch.randn(wl.n_seq, wl.T, wl.n_q, wl.head_dim, generator=g, device="cuda")
    if wl.q_dtype == "bf16":
        q = q.to(torch.bfloat16)
    sinks = torch.randn(wl.n_q, generator=g, device="cuda") if wl.sinks else None
    ref = c.decode(q, sinks=sinks)
    got = _noalloc(c, q, sinks)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert c.device_error() == 0
