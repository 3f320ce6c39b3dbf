"""Parity at the full sizes of the five decode workloads, in the launch
configuration the benchmark times (automatic kernel choice, default query
bits), against the fp64 oracle on the same seeded host inputs.

Every sequence of batch64 and every verify round of spec_verify is checked;
the ring growth (swa_ring) is checked at chosen lengths, since the oracle
would otherwise redo 131072 decodes.  Append bytes of every row checked are
compared exactly."""

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_08_gb300.cache import KVCache
from quantized_kv_cache_08_gb300.inputs import workload
from tests.kvq_testutil import assert_close, need_gpu, oracle_input, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _rows_equal(cache, seq, lo, hi, k_ref, v_ref, what):
    plo, phi = cache.physical_rows(seq, lo, hi)
    kd = cache.k_rows(seq, plo, phi).cpu().numpy()
    vd = cache.v_rows(seq, plo, phi).cpu().numpy()
    assert np.array_equal(kd, k_ref), f"{what}: K bytes differ"
    assert np.array_equal(vd, v_ref), f"{what}: V bytes differ"


def _prefill(cache, wl, seq, n, chunk=64):
    k, v = wl.kv(seq, 0, n)
    kd, vd = to_dev(k), to_dev(v)
    for t0 in range(0, n, chunk):
        t1 = min(n, t0 + chunk)
        cache.append(kd[t0:t1].unsqueeze(0), vd[t0:t1].unsqueeze(0), seq_ids=[seq])
    return k, v


def test_ctx32k_full():
    """32768 rows, 32 Q / 8 KV heads, 1% outlier channels, bf16 q: every row's
    bytes and every output of the T=1 decode."""
    wl = workload("ctx32k")
    L = wl.lengths()[0]
    c = KVCache(1, wl.n_kv, wl.head_dim, wl.n_q, max_t=64, max_rows=L)
    k, v = _prefill(c, wl, 0, L)
    kq = O.quantize_k_rows(k.numpy(), wl.n_kv, wl.head_dim)
    vq = O.quantize_v_rows(v.numpy(), wl.n_kv, wl.head_dim)
    _rows_equal(c, 0, 0, L, kq, vq, "ctx32k")
    q = wl.q(0)
    got = c.decode(to_dev(q)).cpu().numpy()
    ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim)
    ora.append_bytes(0, kq, vq)
    ref = ora.decode(oracle_input(q))
    assert_close(got, ref, what="ctx32k decode")
    assert c.device_error() == 0


def test_ctx32k_full_e4m3():
    """The 32k workload with FP8 E4M3 K/V planes (stream-K kernel): every
    row's bytes and every output of the T=1 decode."""
    wl = workload("ctx32k")
    L = wl.lengths()[0]
    c = KVCache(1, wl.n_kv, wl.head_dim, wl.n_q, max_t=64, max_rows=L, fmt="e4m3")
    k, v = _prefill(c, wl, 0, L)
    ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim, fmt="e4m3")
    ora.append(k.numpy()[None], v.numpy()[None])
    ko, vo = ora.rows(0, 0, L)
    _rows_equal(c, 0, 0, L, ko, vo, "ctx32k e4m3")
    q = wl.q(0)
    got = c.decode(to_dev(q)).cpu().numpy()
    ref = ora.decode(oracle_input(q))
    assert_close(got, ref, what="ctx32k e4m3 decode")
    assert c.device_error() == 0


def test_batch64_all_sequences():
    """64 ragged sequences (prefill len-1, one appended row each, T=1
    decode): every sequence byte for byte and output for output."""
    wl = workload("batch64")
    lens = wl.lengths()
    c = KVCache(wl.n_seq, wl.n_kv, wl.head_dim, wl.n_q, max_t=64, max_rows=max(lens))
    for b, L in enumerate(lens):
        _prefill(c, wl, b, L - 1)
    knew = torch.stack([wl.kv(b, L - 1, L)[0] for b, L in enumerate(lens)])
    vnew = torch.stack([wl.kv(b, L - 1, L)[1] for b, L in enumerate(lens)])
    c.append(to_dev(knew), to_dev(vnew))                  # one row per sequence
    assert c.lens() == lens
    q = wl.q(0)
    got = c.decode(to_dev(q)).cpu().numpy()
    for b, L in enumerate(lens):
        k, v = wl.kv(b, 0, L)
        kq = O.quantize_k_rows(k.numpy(), wl.n_kv, wl.head_dim)
        vq = O.quantize_v_rows(v.numpy(), wl.n_kv, wl.head_dim)
        _rows_equal(c, b, 0, L, kq, vq, f"batch64 seq {b}")
        ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim)
        ora.append_bytes(0, kq, vq)
        ref = ora.decode(oracle_input(q[b:b + 1]))
        assert_close(got[b:b + 1], ref, what=f"batch64 seq {b} (len {L})")
    assert c.device_error() == 0


def _ring_checkpoints(n, window, cap, seed):
    pts = {1, 2, 31, 32, 33, window - 1, window, window + 1, cap, cap + 1, cap + 2, 8192,
           65536, n}
    # the steps either side of the first five rebases: a rebase happens when
    # the appended row would overflow the ring, i.e. at len = cap + 32 j (+1)
    for j in range(5):
        for d in (-1, 0, 1, 2):
            pts.add(cap + 32 * j + d)
    rng = np.random.default_rng(seed)
    pts.update(int(x) for x in rng.integers(1, n + 1, size=32))
    return sorted(p for p in pts if 1 <= p <= n)


def test_swa_ring_growth_to_131072():
    """64 Q / 8 KV heads, head_dim 64, sinks, window 4096 over a ring of
    window + 31 rows, T=1 appends until the length is 131072; at chosen
    lengths the live rows equal the oracle's bytes and the decode matches
    the windowed oracle."""
    wl = workload("swa_ring")
    N, W = wl.lengths()[0], wl.window
    c = KVCache(1, wl.n_kv, wl.head_dim, wl.n_q, max_t=1, window=W, ring=True)
    cap = c.rows
    assert cap == W + 31
    k, v = wl.kv(0, 0, N)
    kq = O.quantize_k_rows(k.numpy(), wl.n_kv, wl.head_dim)
    vq = O.quantize_v_rows(v.numpy(), wl.n_kv, wl.head_dim)
    kd, vd = to_dev(k), to_dev(v)
    sinks = wl.sink_logits()
    sinks_d = to_dev(sinks)
    checks = set(_ring_checkpoints(N, W, cap, seed=4))
    n_checked = 0
    for t in range(N):
        c.append(kd[t:t + 1].view(1, 1, wl.n_kv, wl.head_dim), vd[t:t + 1].view(1, 1, wl.n_kv, wl.head_dim))
        L = t + 1
        if L not in checks:
            continue
        base = c.bases()[0]
        lstart = max(0, L - W)
        assert base <= lstart and lstart - base <= 31 and L - base <= cap, (L, base)
        _rows_equal(c, 0, max(base, lstart), L, kq[max(base, lstart):L], vq[max(base, lstart):L],
                    f"ring len {L}")
        q = wl.q(L)
        got = c.decode(to_dev(q), sinks=sinks_d).cpu().numpy()
        # rows before lstart are invisible: the oracle holds the window suffix
        ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim, window=W)
        ora.append_bytes(0, kq[lstart:L], vq[lstart:L])
        ref = ora.decode(oracle_input(q), sinks=sinks.double().numpy())
        assert_close(got, ref, what=f"ring decode at len {L}")
        n_checked += 1
    assert n_checked >= 40
    assert c.lens() == [N]
    assert c.device_error() == 0


def test_spec_verify_100_rounds():
    """16 Q / 4 KV heads, head_dim 256, 16384 rows, then 100 rounds of append
    T=8, causal T=8 decode, truncate to snapshot + accept: the 8 appended
    rows' bytes and all outputs, every round."""
    wl = workload("spec_verify")
    L0, T, R = wl.lengths()[0], wl.T, wl.rounds
    c = KVCache(1, wl.n_kv, wl.head_dim, wl.n_q, max_t=64, max_rows=L0 + T * (R + 1))
    ora = O.OracleKvCache(1, wl.n_kv, wl.head_dim)
    k, v = _prefill(c, wl, 0, L0)
    ora.append(k.unsqueeze(0).numpy(), v.unsqueeze(0).numpy())
    accepts = wl.accepts()
    snap = L0
    for r in range(R):
        # draft rows of round r: a deterministic stream per round
        kr, vr = wl.kv(1 + r, 0, T)
        c.append(to_dev(kr).unsqueeze(0), to_dev(vr).unsqueeze(0))
        ora.append(kr.unsqueeze(0).numpy(), vr.unsqueeze(0).numpy())
        ko, vo = ora.rows(0, snap, snap + T)
        _rows_equal(c, 0, snap, snap + T, ko, vo, f"round {r}")
        q = wl.q(r)
        got = c.decode(to_dev(q)).cpu().numpy()
        ref = ora.decode(oracle_input(q))
        assert_close(got, ref, what=f"verify round {r}")
        snap += accepts[r]
        c.truncate([snap])
        ora.truncate([snap])
        assert c.lens() == [snap]
    assert c.device_error() == 0
