"""GPU parity of the FP8 E4M3 K/V format (one byte per element, no scale)
through the C ABI against the fp64 oracle.

Append bytes must be bit-exact, including rounding ties, subnormals, signed
zeros and saturation beyond 448; attention outputs must be within 2e-3 max abs
error of the oracle run on the same bytes (both kernels decode E4M3 exactly
and compute in fp32, so the error is far below that).  E4M3 caches decode on
the stream-K kernel where its geometry allows (head_dim 64, 128 or 256, token
rows of 16-byte multiples), else on the generic split kernel."""

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from tests.kvq_testutil import Pair, assert_close, assert_rows_equal, need_gpu, oracle_input, to_dev
from quantized_kv_cache_08_gb300 import _binding as B
from quantized_kv_cache_08_gb300.cache import KVCache

pytestmark = pytest.mark.gpu

F8 = "e4m3"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _randn(*shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g) * scale


@pytest.mark.parametrize("n_kv,D,T,dtype,scale", [
    (2, 128, 1, torch.float32, 1.0), (2, 128, 7, torch.float32, 40.0), (8, 64, 3, torch.float32, 1e-2),
    (1, 32, 5, torch.bfloat16, 100.0), (4, 256, 2, torch.bfloat16, 1.0), (3, 96, 4, torch.float32, 3.0),
])
def test_fp8_append_bytes_exact(n_kv, D, T, dtype, scale):
    """Random rows (scale 40 and 100 push many elements past 448, 1e-2 into
    the subnormals), bf16 inputs and a permuted subset of sequences."""
    B_ = 3
    p = Pair(B_, n_kv, D, n_kv * 2, max_t=T, max_rows=64, fmt=F8)
    assert p.dev.k_tok == p.dev.v_tok == n_kv * D
    for step in range(4):
        k = _randn(B_, T, n_kv, D, seed=10 * step + 1, scale=scale).to(dtype)
        v = _randn(B_, T, n_kv, D, seed=10 * step + 2, scale=0.5 * scale).to(dtype) + 1.0
        p.append(k, v)
    k = _randn(2, T, n_kv, D, seed=99, scale=scale).to(dtype)
    p.append(k, -k, seq_ids=[2, 0])
    assert p.dev.lens() == [5 * T, 4 * T, 5 * T]
    for b in range(B_):
        assert_rows_equal(p.dev, p.ora, b, 0, p.dev.lens()[b])
    assert p.dev.device_error() == 0


def test_fp8_append_ties_subnormals_zeros_and_saturation():
    """Every midpoint between adjacent E4M3 values (and its float32
    neighbours), every representable value, signed zeros and values at and
    beyond the largest finite 448."""
    grid = O.e4m3_value(np.arange(0x7F)).astype(np.float32)   # 0 .. 448
    mids = ((grid[1:].astype(np.float64) + grid[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([
        grid, -grid, mids, -mids,
        np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf)),
        np.array([0.0, -0.0, 448.0, 463.99, 464.0, 464.01, 480.0, 1e6, -1e6, 3e38, -3e38,
                  2.0 ** -10, -(2.0 ** -10), 2.0 ** -12, 1e-30], np.float32),
    ]).astype(np.float32)
    n = -(-vals.size // 32) * 32
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.float32)])
    x = torch.from_numpy(vals.reshape(-1, 1, 1, 32))
    p = Pair(x.shape[0], 1, 32, 1, max_rows=2, fmt=F8)
    p.append(x, -x)
    for b in range(x.shape[0]):
        assert_rows_equal(p.dev, p.ora, b, 0, 1)
    # the bytes decode to the values of the oracle's table
    k = p.dev.k_rows(0, 0, 1).cpu().numpy()
    np.testing.assert_array_equal(O.e4m3_value(k[0]), O.e4m3_value(O.e4m3_bits(vals[:32])))


CASES = [
    # B, Hq, Hkv, D, lens, T, window, ring, sinks, qdtype
    (1, 8, 2, 128, [512], 1, 0, False, False, torch.float32),
    (3, 32, 8, 128, [1000, 1, 333], 1, 0, False, False, torch.float32),
    (2, 32, 8, 128, [700, 2049], 1, 0, False, True, torch.bfloat16),
    (1, 64, 8, 64, [600], 1, 128, False, True, torch.float32),
    (2, 16, 4, 256, [300, 77], 8, 50, False, True, torch.float32),
    (2, 16, 8, 32, [130, 64], 3, 0, False, True, torch.float32),
    (4, 8, 2, 128, [5, 17, 64, 65], 4, 0, False, True, torch.float32),
    (2, 4, 1, 128, [300, 45], 1, 0, False, True, torch.float32),
]


@pytest.mark.parametrize("path", [0, 1, 2, 3], ids=["auto", "generic", "stream", "stream_rs2"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8_decode_matches_oracle(case, path):
    Bn, Hq, Hkv, D, lens, T, window, ring, sinks, qdt = case
    p = Pair(Bn, Hkv, D, Hq, max_t=max(T, 64), max_rows=max(lens) + T, window=window, ring=ring, fmt=F8)
    p.dev.set_decode_path(min(path, 2))
    p.dev.set_row_slices(2 if path == 3 else 0)
    if path >= 2 and (D not in (64, 128, 256) or (Hkv * D) % 16):
        p.append(_randn(Bn, 1, Hkv, D, seed=1), _randn(Bn, 1, Hkv, D, seed=2))
        with pytest.raises(B.KvqError) as e:
            p.dev.decode(to_dev(_randn(Bn, 1, Hq, D, seed=3)))
        assert e.value.status == B.KVQ_EUNSUPPORTED
        return
    for b, L in enumerate(lens):
        k = _randn(1, L, Hkv, D, seed=100 + b, scale=2.0)
        v = _randn(1, L, Hkv, D, seed=200 + b)
        for t0 in range(0, L, 64):
            p.append(k[:, t0:t0 + 64], v[:, t0:t0 + 64], seq_ids=[b])
    q = _randn(Bn, T, Hq, D, seed=7).to(qdt)
    s = _randn(Hq, seed=8) if sinks else None
    got, ref = p.decode(q, sinks=s)
    err = assert_close(got, ref)
    assert err <= 1e-4, f"fp32-level path error {err:.2e}"
    assert p.dev.device_error() == 0


def test_fp8_stream_kernel_equals_generic_and_refuses_head_dim_32():
    """Forced onto the stream-K kernel an E4M3 cache gives the generic
    kernel's result to fp32 rounding; a head_dim it does not take is refused."""
    p = Pair(2, 8, 128, 32, max_t=64, max_rows=700, fmt=F8)
    for b, L in enumerate((640, 333)):
        k = _randn(1, L, 8, 128, seed=5 + b, scale=3.0)
        for t0 in range(0, L, 64):
            p.append(k[:, t0:t0 + 64], -k[:, t0:t0 + 64], seq_ids=[b])
    q = to_dev(_randn(2, 1, 32, 128, seed=6))
    p.dev.set_decode_path(2)
    stream = p.dev.decode(q).cpu().numpy()
    p.dev.set_decode_path(1)
    generic = p.dev.decode(q).cpu().numpy()
    assert np.max(np.abs(stream - generic)) <= 1e-5
    small = Pair(1, 4, 32, 8, max_t=8, max_rows=64, fmt=F8)
    small.append(_randn(1, 8, 4, 32, seed=7), _randn(1, 8, 4, 32, seed=8))
    small.dev.set_decode_path(2)
    with pytest.raises(B.KvqError) as e:
        small.dev.decode(to_dev(_randn(1, 1, 8, 32, seed=9)))
    assert e.value.status == B.KVQ_EUNSUPPORTED
    assert p.dev.device_error() == 0


@pytest.mark.parametrize("split_rows", [64, 200, 1000])
def test_fp8_split_sizes_agree(split_rows):
    Hq, Hkv, D, L = 32, 8, 128, 3000
    p = Pair(2, Hkv, D, Hq, max_t=64, max_rows=L, fmt=F8)
    for b in range(2):
        k = _randn(1, L - 100 * b, Hkv, D, seed=300 + b)
        for t0 in range(0, k.shape[1], 64):
            p.append(k[:, t0:t0 + 64], 0.5 * k[:, t0:t0 + 64], seq_ids=[b])
    p.dev.set_decode_path(1)                    # split sizes belong to the generic kernel
    p.dev.set_split_rows(split_rows)
    got, ref = p.decode(_randn(2, 1, Hq, D, seed=9))
    assert_close(got, ref)


def test_fp8_ring_growth_and_truncate_match_oracle():
    """A ring (window 64) grown past several rebases with T = 1 steps, then a
    rollback and re-append: live bytes and outputs follow the oracle."""
    Hq, Hkv, D, W, N = 16, 4, 64, 64, 400
    p = Pair(1, Hkv, D, Hq, max_t=1, window=W, ring=True, fmt=F8)
    k = _randn(1, N, Hkv, D, seed=91)
    v = _randn(1, N, Hkv, D, seed=92)
    s = _randn(Hq, seed=93)
    for t in range(N):
        p.append(k[:, t:t + 1], v[:, t:t + 1])
        L = t + 1
        if t % 9 == 0 or t > N - 3:
            got, ref = p.decode(_randn(1, 1, Hq, D, seed=1000 + t), sinks=s)
            assert_close(got, ref, what=f"step {t}")
            base = p.dev.bases()[0]
            assert_rows_equal(p.dev, p.ora, 0, max(base, L - W), L)
    assert p.dev.bases()[0] > 0
    p.truncate([N - 5])
    p.append(k[:, :1], -v[:, :1])
    got, ref = p.decode(_randn(1, 1, Hq, D, seed=5000), sinks=s)
    assert_close(got, ref)
    assert p.dev.device_error() == 0


def test_fp8_softcap_and_noalloc_decode():
    """Score soft-capping and the no-alloc entry point on an E4M3 cache."""
    Hq, Hkv, D, L = 32, 8, 128, 900
    p = Pair(1, Hkv, D, Hq, max_t=64, max_rows=L, fmt=F8)
    k = _randn(1, L, Hkv, D, seed=61)
    v = _randn(1, L, Hkv, D, seed=62)
    for t0 in range(0, L, 64):
        p.append(k[:, t0:t0 + 64], v[:, t0:t0 + 64])
    q = _randn(1, 1, Hq, D, seed=63, scale=4.0)
    p.dev.set_softcap(3.0)
    got = p.dev.decode(to_dev(q)).cpu().numpy()
    ref = p.ora.decode(oracle_input(q), softcap=3.0)
    assert_close(got, ref, what="softcap 3")
    p.dev.set_softcap(0.0)
    plain = p.dev.decode(to_dev(q))
    out = torch.empty_like(plain)
    qd = to_dev(q)
    B.kvq_decode_noalloc(p.dev.handle, qd.data_ptr(), B.KVQ_F32, 1, Hq, None, 0.0, out.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    assert torch.equal(out, plain)
    assert_close(plain.cpu().numpy(), p.ora.decode(oracle_input(q)))


def test_fp8_captured_append_decode_replays():
    Hq, Hkv, D, L0, steps = 32, 8, 128, 500, 12
    p = Pair(1, Hkv, D, Hq, max_t=64, max_rows=L0 + steps + 1, fmt=F8)
    k = _randn(1, L0 + steps + 1, Hkv, D, seed=101)
    v = _randn(1, L0 + steps + 1, Hkv, D, seed=102)
    for t0 in range(0, L0, 64):
        p.append(k[:, t0:min(L0, t0 + 64)], v[:, t0:min(L0, t0 + 64)])
    kd, vd = to_dev(k), to_dev(v)
    k_in = torch.empty(1, 1, Hkv, D, device="cuda")
    v_in = torch.empty_like(k_in)
    q_in = torch.zeros(1, 1, Hq, D, device="cuda")
    out = torch.empty(1, 1, Hq, D, device="cuda")
    k_in.copy_(kd[:, L0:L0 + 1])
    v_in.copy_(vd[:, L0:L0 + 1])
    p.dev.append(k_in, v_in)
    p.dev.decode(q_in, out=out)
    p.dev.truncate([L0])
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        p.dev.append(k_in, v_in)
        p.dev.decode(q_in, out=out)
    p.dev.note_replayed(0, 1)
    p.dev.truncate([L0])
    for t in range(steps):
        q = _randn(1, 1, Hq, D, seed=2000 + t)
        k_in.copy_(kd[:, L0 + t:L0 + t + 1])
        v_in.copy_(vd[:, L0 + t:L0 + t + 1])
        q_in.copy_(to_dev(q))
        g.replay()
        p.dev.note_replayed(1, 1)
        p.ora.append(k[:, L0 + t:L0 + t + 1].numpy(), v[:, L0 + t:L0 + t + 1].numpy())
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), p.ora.decode(q.double().numpy()), what=f"replay {t}")
    assert_rows_equal(p.dev, p.ora, 0, 0, L0 + steps)
