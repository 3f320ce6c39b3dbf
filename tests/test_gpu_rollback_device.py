"""GPU parity of the rollback whose accepted counts stay on the device
(kvq_truncate_device): speculative-decode rounds of append T draft rows,
decode the T causal rows, keep accept[b] of them, against the oracle's
rollback (len = snapshot_len + accept_len).  Covers the host's bounded
mirror, a device-side refusal of bad counts, a ring whose rebases need a
length read-back, and a whole round captured in a CUDA graph."""

import numpy as np
import pytest
import torch

from tests.kvq_testutil import Pair, assert_close, assert_rows_equal, need_gpu, to_dev
from quantized_kv_cache_08_gb300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _randn(*shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g) * scale


def _prefill(p, lens, Hkv, D, seed, chunk=64):
    for b, L in enumerate(lens):
        k = _randn(1, L, Hkv, D, seed=seed + b)
        v = _randn(1, L, Hkv, D, seed=seed + 50 + b)
        for t0 in range(0, L, chunk):
            p.append(k[:, t0:t0 + chunk], v[:, t0:t0 + chunk], seq_ids=[b])


@pytest.mark.parametrize("fmt", ["q8_0/q5_1", "e4m3"])
def test_device_rollback_rounds_match_oracle(fmt):
    Bn, Hq, Hkv, D, T, rounds = 3, 16, 4, 128, 8, 12
    lens = [300, 41, 1000]
    p = Pair(Bn, Hkv, D, Hq, max_t=64, max_rows=max(lens) + (rounds + 1) * T, fmt=fmt)
    _prefill(p, lens, Hkv, D, seed=10)
    rng = np.random.default_rng(5)
    acc_d = torch.zeros(Bn, dtype=torch.int32, device="cuda")
    for r in range(rounds):
        k = _randn(Bn, T, Hkv, D, seed=100 + r)
        v = _randn(Bn, T, Hkv, D, seed=200 + r)
        p.append(k, v)
        got, ref = p.decode(_randn(Bn, T, Hq, D, seed=300 + r))
        assert_close(got, ref, what=f"round {r}")
        acc = rng.integers(0, T + 1, Bn)
        acc_d.copy_(torch.from_numpy(acc.astype(np.int32)))
        p.dev.truncate_device(acc_d, T)
        p.ora.rollback(acc, T)
        if r % 4 == 3:
            p.dev.sync_len()
            assert p.dev.lens() == p.ora.lens()
    # one T=1 decode straight after a rollback, before any read-back
    got, ref = p.decode(_randn(Bn, 1, Hq, D, seed=400))
    assert_close(got, ref, what="after rollback")
    p.dev.sync_len()
    assert p.dev.lens() == p.ora.lens()
    for b in range(Bn):
        assert_rows_equal(p.dev, p.ora, b, 0, p.ora.lens()[b])
    assert p.dev.device_error() == 0


def test_device_rollback_refuses_bad_counts_and_keeps_host_bounds():
    Hkv, D, Hq, T = 2, 64, 4, 4
    p = Pair(3, Hkv, D, Hq, max_t=8, max_rows=64)
    _prefill(p, [20, 20, 20], Hkv, D, seed=30, chunk=8)
    p.append(_randn(3, T, Hkv, D, seed=31), _randn(3, T, Hkv, D, seed=32))
    # 5 > T and -1 are refused on the device: those sequences keep 24 rows
    acc_d = torch.tensor([5, -1, 2], dtype=torch.int32, device="cuda")
    p.dev.truncate_device(acc_d, T)
    assert p.dev.device_error() == 1
    p.dev.sync_len()
    assert p.dev.lens() == [24, 24, 22]
    p.ora.truncate([24, 24, 22])
    # while a rollback is pending the host knows each length within [len - T, len]
    p.append(_randn(3, T, Hkv, D, seed=33), _randn(3, T, Hkv, D, seed=34))
    p.dev.truncate_device(torch.zeros(3, dtype=torch.int32, device="cuda"), T)
    p.ora.rollback([0, 0, 0], T)
    assert p.dev.lens() == [28, 28, 26]                 # upper ends
    with pytest.raises(B.KvqError) as e:
        p.dev.truncate([25, 24, 22])                    # above the lower end of sequence 0
    assert e.value.status == B.KVQ_ERANGE
    p.truncate([24, 23, 22])                            # within the lower ends: exact again
    assert p.dev.lens() == [24, 23, 22]
    for b in range(3):
        assert_rows_equal(p.dev, p.ora, b, 0, p.ora.lens()[b])
    got, ref = p.decode(_randn(3, 1, Hq, D, seed=35))
    assert_close(got, ref)
    # a sequence that may hold fewer than T rows is refused on the host
    q = Pair(1, Hkv, D, Hq, max_t=8, max_rows=16)
    q.append(_randn(1, 2, Hkv, D, seed=36), _randn(1, 2, Hkv, D, seed=37))
    with pytest.raises(B.KvqError) as e:
        q.dev.truncate_device(torch.zeros(1, dtype=torch.int32, device="cuda"), 4)
    assert e.value.status == B.KVQ_ERANGE
    assert p.dev.device_error() == 0 and q.dev.device_error() == 0


def test_ring_device_rollback_reads_lengths_back_before_a_rebase():
    """Draft rounds on a window ring: an append that would rebase while a
    rollback is pending is refused until kvq_sync_len; outputs and live rows
    follow the windowed oracle throughout."""
    Hq, Hkv, D, W, T, rounds = 16, 4, 64, 128, 8, 90
    p = Pair(1, Hkv, D, Hq, max_t=T, window=W, ring=True)
    assert p.dev.rows == W + 30 + T
    _prefill(p, [100], Hkv, D, seed=40, chunk=T)
    rng = np.random.default_rng(41)
    acc_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    refused = 0
    for r in range(rounds):
        k = _randn(1, T, Hkv, D, seed=500 + r)
        v = _randn(1, T, Hkv, D, seed=600 + r)
        try:
            p.append(k, v)
        except B.KvqError as e:
            assert e.status == B.KVQ_ERANGE
            refused += 1
            p.dev.sync_len()
            p.append(k, v)
        got, ref = p.decode(_randn(1, T, Hq, D, seed=700 + r))
        assert_close(got, ref, what=f"round {r}")
        a = int(rng.integers(0, T + 1))
        acc_d.fill_(a)
        p.dev.truncate_device(acc_d, T)
        p.ora.rollback([a], T)
    p.dev.sync_len()
    L = p.ora.lens()[0]
    assert p.dev.lens() == [L]
    base = p.dev.bases()[0]
    assert refused > 0 and base > 0
    assert_rows_equal(p.dev, p.ora, 0, max(base, L - W), L)
    assert p.dev.device_error() == 0


def test_captured_draft_round_with_device_rollback_replays():
    """append T draft rows + T-row decode + device-side rollback captured once
    as a CUDA graph and replayed with a new accepted count each round."""
    Hq, Hkv, D, L0, T, rounds = 32, 8, 128, 1000, 4, 10
    p = Pair(1, Hkv, D, Hq, max_t=64, max_rows=L0 + (rounds + 2) * T)
    _prefill(p, [L0], Hkv, D, seed=50)
    k_in = torch.empty(1, T, Hkv, D, device="cuda")
    v_in = torch.empty_like(k_in)
    q_in = torch.zeros(1, T, Hq, D, device="cuda")
    out = torch.empty(1, T, Hq, D, device="cuda")
    acc_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    # warm up outside the capture, accepting nothing
    k_in.zero_()
    v_in.zero_()
    p.dev.append(k_in, v_in)
    p.dev.decode(q_in, out=out)
    p.dev.truncate_device(acc_d, T)
    p.dev.sync_len()
    assert p.dev.lens() == [L0]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        p.dev.append(k_in, v_in)
        p.dev.decode(q_in, out=out)
        p.dev.truncate_device(acc_d, T)
    p.dev.sync_len()                                    # the capture ran nothing
    assert p.dev.lens() == [L0]
    rng = np.random.default_rng(51)
    for r in range(rounds):
        k = _randn(1, T, Hkv, D, seed=800 + r)
        v = _randn(1, T, Hkv, D, seed=900 + r)
        q = _randn(1, T, Hq, D, seed=1000 + r)
        a = int(rng.integers(0, T + 1))
        k_in.copy_(to_dev(k))
        v_in.copy_(to_dev(v))
        q_in.copy_(to_dev(q))
        acc_d.fill_(a)
        g.replay()
        p.ora.append(k.numpy(), v.numpy())
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), p.ora.decode(q.double().numpy()), what=f"replay {r}")
        p.ora.rollback([a], T)
    p.dev.sync_len()
    assert p.dev.lens() == p.ora.lens()
    assert_rows_equal(p.dev, p.ora, 0, 0, p.ora.lens()[0])
    assert p.dev.device_error() == 0
