"""Pins of the fp64 oracle against things other than itself.

* binary16 encoding: numpy's float16 cast (a library routine) on a million
  doubles and on every midpoint, plus hand-derived encodings fixed by IEEE 754;
* q8_0 / q5_1 bytes: hand-derived blocks (tests/golden), an independent exact
  rational-arithmetic quantiser (fractions.Fraction), and the round-trip
  bounds |x - x_hat| <= d/2;
* FP8 E4M3 bytes: hand-derived encodings (tests/golden), torch's
  float8_e4m3fn decoding of every byte and encoding of in-range values (library
  routines), and a brute-force nearest-value search over the finite codes;
* attention: torch's scaled_dot_product_attention in float64 (an independent
  library routine) with the sink written as an extra value-less column and the
  window / causal rules written as an additive -inf mask, plus closed forms
  (one row, q = 0) and the invariants the pages state (GQA = repeated KV heads,
  T-row causal = sequential append-then-attend, window >= len = full).
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _parse_float(tok):
    return float.fromhex(tok) if tok.lstrip("-").startswith("0x") else float(tok)


def _golden(name):
    out = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.split()
    return out


# ---------------------------------------------------------------- binary16

def test_f16_known_encodings():
    with open(os.path.join(GOLD, "f16_known.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    vals = np.array([_parse_float(r[0]) for r in rows])
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint16)
    np.testing.assert_array_equal(O.f16_bits(vals), want)


def test_f16_matches_numpy_random():
    rng = np.random.default_rng(1)
    # exponents spread over subnormal, normal and overflow ranges
    mant = rng.uniform(1.0, 2.0, 1_000_000)
    ex = rng.integers(-30, 18, 1_000_000)
    y = np.ldexp(mant, ex) * rng.choice([-1.0, 1.0], 1_000_000)
    with np.errstate(over="ignore"):
        ref = y.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.f16_bits(y), ref)


def test_f16_matches_numpy_on_every_midpoint():
    # every pair of adjacent finite binary16 values, its midpoint, and one
    # float64 ulp either side of the midpoint
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).view(np.float16).astype(np.float64)
    mid = (a + b) / 2
    ys = np.concatenate([mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf),
                         -mid, a, -b])
    with np.errstate(over="ignore"):
        ref = ys.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.f16_bits(ys), ref)


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.f16_value(bits)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isinf(got[np.isinf(ref)]))
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_round_half_away():
    t = np.array([0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.49999999999999994, -0.0,
                  2.4999999999999996, 126.5, 3.0])
    np.testing.assert_array_equal(
        O.round_half_away(t), [1, -1, 2, -2, 3, -3, 0, 0, 2, 127, 3])


# ------------------------------------------------- exact rational reference
# An independent quantiser in exact rational arithmetic: binary16 rounding of
# a Fraction is done with integer arithmetic, codes with exact comparisons.

def _f16_round_fraction(r: Fraction) -> Fraction:
    """Nearest binary16 value to the exact rational r >= 0, ties to even."""
    assert r >= 0
    if r == 0:
        return Fraction(0)
    e = r.numerator.bit_length() - r.denominator.bit_length()
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    e = max(e, -14)
    q = Fraction(2) ** (e - 10)
    n = r / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * q
    assert v <= 65504, "overflow not expected in these tests"
    return v


def _rha_fraction(t: Fraction) -> int:
    a = abs(t)
    fl = a.numerator // a.denominator
    if a - fl >= Fraction(1, 2):
        fl += 1
    return fl if t >= 0 else -fl


def _exact_q8_0(x32):
    xs = [Fraction(float(v)) for v in x32]
    amax = max(abs(v) for v in xs)
    d = _f16_round_fraction(amax / 127)
    codes = [0] * 32 if d == 0 else [max(-127, min(127, _rha_fraction(v / d))) for v in xs]
    return d, codes


def _exact_q5_1(x32):
    xs = [Fraction(float(v)) for v in x32]
    mn, mx = min(xs), max(xs)
    d = _f16_round_fraction((mx - mn) / 31)
    m = _f16_round_fraction(abs(mn)) * (1 if mn >= 0 else -1)
    u = [0] * 32 if d == 0 else [max(0, min(31, _rha_fraction((v - m) / d))) for v in xs]
    return d, m, u


def _blocks(rng, n):
    """Random float32 blocks with varied scale, a few adversarial ones."""
    x = rng.standard_normal((n, 32)).astype(np.float32)
    x *= np.float32(10.0) ** rng.integers(-3, 3, (n, 1)).astype(np.float32)
    return x


def test_q8_0_matches_exact_rationals():
    rng = np.random.default_rng(7)
    x = _blocks(rng, 300)
    # adversarial scales: amax = 127 * (binary16 midpoint) and one fp32 ulp
    # either side, so that a double rounding of amax/127 would show
    adv = []
    for mid_bits in (0x3C00, 0x2E66, 0x0400, 0x0123, 0x5555):
        lo = np.array(mid_bits, np.uint16).view(np.float16).astype(np.float64)
        hi = np.array(mid_bits + 1, np.uint16).view(np.float16).astype(np.float64)
        amax = np.float32(127.0 * (lo + hi) / 2)
        for a in (amax, np.nextafter(amax, np.float32(0)), np.nextafter(amax, np.float32(np.inf))):
            blk = rng.standard_normal(32).astype(np.float32)
            blk = blk / np.max(np.abs(blk)) * a * np.float32(0.9)
            blk[5] = a
            adv.append(blk)
    x = np.concatenate([x, np.array(adv, np.float32)])
    # exact ties of the codes: x = (n + 1/2) d
    tie = np.zeros((1, 32), np.float32)
    tie[0, 0] = 127.0
    tie[0, 1:] = (np.arange(31) - 15 + 0.5).astype(np.float32)
    x = np.concatenate([x, tie])
    got = O.q8_0_quantize(x)
    for i in range(x.shape[0]):
        d, codes = _exact_q8_0(x[i])
        gd, gc = O.q8_0_fields(got[i])
        assert Fraction(float(gd)) == d, i
        assert list(gc) == codes, i


def test_q5_1_matches_exact_rationals():
    rng = np.random.default_rng(8)
    x = _blocks(rng, 300)
    x[:20] += np.float32(50.0)            # all-positive blocks
    x[20:40] -= np.float32(50.0)          # all-negative blocks
    got = O.q5_1_quantize(x)
    for i in range(x.shape[0]):
        d, m, u = _exact_q5_1(x[i])
        gd, gm, gu = O.q5_1_fields(got[i])
        assert Fraction(float(gd)) == d, i
        assert Fraction(float(gm)) == m, i
        assert list(gu) == u, i


# ---------------------------------------------------------- hand-derived

def test_q5_1_ramp_golden():
    g = _golden("q5_1_ramp.txt")
    x = np.array([float(t) for t in g["input"]], np.float32)
    want = bytes(int(t, 16) for t in g["bytes"])
    assert O.q5_1_quantize(x).tobytes() == want
    np.testing.assert_array_equal(O.q5_1_dequantize(np.frombuffer(want, np.uint8)), x)


def test_q8_0_unit_scale_golden():
    g = _golden("q8_0_unit_scale.txt")
    x = np.array([float(t) for t in g["input"]], np.float32)
    codes = np.array([int(t) for t in g["codes"]], np.int8)
    blk = O.q8_0_quantize(x)
    assert int(blk[0]) | (int(blk[1]) << 8) == int(g["d_bits"][0], 16)
    np.testing.assert_array_equal(blk[2:].view(np.int8), codes)


def test_block_sizes_and_zero_blocks():
    z = np.zeros((3, 32), np.float32)
    assert O.q8_0_quantize(z).shape == (3, 34)
    assert O.q5_1_quantize(z).shape == (3, 24)
    assert not O.q8_0_quantize(z).any()
    assert not O.q5_1_quantize(z).any()
    # constant block: d = 0, u = 0, x_hat = fp16(x)
    c = np.full(32, 0.1, np.float32)
    blk = O.q5_1_quantize(c)
    d, m, u = O.q5_1_fields(blk)
    assert d == 0 and not u.any()
    assert m == np.float32(0.1).astype(np.float16).astype(np.float64)


def test_round_trip_bounds():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4000, 32)).astype(np.float32)
    x[:, 3] *= 10          # outlier channel, as in the 32k-context workload
    x64 = x.astype(np.float64)
    k = O.q8_0_quantize(x)
    d, c = O.q8_0_fields(k)
    assert np.all(np.abs(c) <= 127)
    assert np.all(np.max(np.abs(c), axis=-1) == 127)
    assert np.all(np.abs(x64 - O.q8_0_dequantize(k)) <= d[:, None] / 2)
    v = O.q5_1_quantize(x)
    d, m, u = O.q5_1_fields(v)
    assert np.all((u >= 0) & (u <= 31))
    assert np.all(u[np.arange(len(x)), np.argmax(x, axis=1)] == 31)
    assert np.all(u[np.arange(len(x)), np.argmin(x, axis=1)] == 0)
    assert np.all(np.abs(x64 - O.q5_1_dequantize(v)) <= d[:, None] / 2)


def test_row_placement():
    # element e = kv_head*head_dim + d lands in block e//32, lane e%32
    n_kv, D = 3, 64
    x = np.zeros((1, n_kv, D), np.float32)
    x[0, 2, 37] = 5.0                       # e = 2*64 + 37 = 165 -> block 5, lane 5
    rows = O.quantize_k_rows(x, n_kv, D)
    blk = rows.reshape(-1, 34)
    assert blk.shape[0] == n_kv * D // 32
    nz = [i for i in range(blk.shape[0]) if blk[i].any()]
    assert nz == [5]
    assert blk[5, 2 + 5].view(np.int8) == 127
    d, _ = O.q8_0_fields(blk[5])
    assert O.dequantize_k_rows(rows, n_kv, D)[0, 2, 37] == 127 * d
    assert abs(127 * d - 5.0) <= d / 2


# ------------------------------------------------------------- attention

def _sdpa_reference(q, kh, vh, *, scale, sinks, window):
    """torch SDPA (float64) for one sequence, the sink as a value-less extra
    column with additive bias = sink, window/causal as an additive -inf mask."""
    T, Hq, D = q.shape
    L, Hkv, _ = kh.shape
    hpk = Hq // Hkv
    K = torch.from_numpy(kh).permute(1, 0, 2).repeat_interleave(hpk, 0)   # [Hq, L, D]
    V = torch.from_numpy(vh).permute(1, 0, 2).repeat_interleave(hpk, 0)
    Q = torch.from_numpy(np.asarray(q, np.float64)).permute(1, 0, 2)     # [Hq, T, D]
    K = torch.cat([K, torch.zeros(Hq, 1, D, dtype=torch.float64)], 1)
    V = torch.cat([V, torch.zeros(Hq, 1, D, dtype=torch.float64)], 1)
    bias = torch.full((Hq, T, L + 1), -math.inf, dtype=torch.float64)
    s0 = L - T
    for t in range(T):
        upto = s0 + t + 1
        lo = max(0, upto - window) if window else 0
        bias[:, t, lo:upto] = 0.0
    if sinks is not None:
        bias[:, :, L] = torch.from_numpy(np.asarray(sinks, np.float64))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        Q.unsqueeze(0), K.unsqueeze(0), V.unsqueeze(0), attn_mask=bias.unsqueeze(0), scale=scale)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("T,Hq,Hkv,D,L,window,use_sink", [
    (1, 8, 2, 64, 50, 0, False),
    (1, 8, 2, 64, 50, 0, True),
    (1, 4, 4, 32, 70, 16, True),
    (4, 8, 2, 64, 40, 0, False),
    (8, 4, 1, 32, 30, 12, True),
    (3, 6, 3, 96, 9, 5, False),
])
def test_attention_matches_sdpa(T, Hq, Hkv, D, L, window, use_sink):
    rng = np.random.default_rng(T * 100 + L)
    kh = rng.standard_normal((L, Hkv, D))
    vh = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((T, Hq, D))
    sinks = rng.standard_normal(Hq) if use_sink else None
    scale = 1.0 / math.sqrt(D)
    got = O.attend(q, kh, vh, sinks=sinks, window=window)
    ref = _sdpa_reference(q, kh, vh, scale=scale, sinks=sinks, window=window)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(11)
    D = 32
    kh = rng.standard_normal((1, 1, D))
    vh = rng.standard_normal((1, 1, D))
    q = rng.standard_normal((1, 2, D))
    out = O.attend(q, kh, vh)
    np.testing.assert_allclose(out[0, 0], vh[0, 0], rtol=0, atol=1e-15)
    sink = np.array([0.7, -1.3])
    out = O.attend(q, kh, vh, sinks=sink)
    s = (kh[0, 0] @ q[0, 1]) / math.sqrt(D)
    np.testing.assert_allclose(out[0, 1], vh[0, 0] / (1 + math.exp(sink[1] - s)), rtol=1e-14)
    # q = 0: uniform weights, output = mean of visible values
    kh = rng.standard_normal((9, 2, D))
    vh = rng.standard_normal((9, 2, D))
    out = O.attend(np.zeros((1, 4, D)), kh, vh, window=4)
    np.testing.assert_allclose(out[0, 3], vh[5:9, 1].mean(0), rtol=1e-13)


def test_attention_invariants():
    rng = np.random.default_rng(12)
    L, Hq, Hkv, D = 40, 8, 2, 64
    kh = rng.standard_normal((L, Hkv, D))
    vh = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((1, Hq, D))
    plain = O.attend(q, kh, vh)
    # a sink of -inf is the plain softmax
    np.testing.assert_array_equal(O.attend(q, kh, vh, sinks=np.full(Hq, -np.inf)), plain)
    # window >= len is full attention
    np.testing.assert_array_equal(O.attend(q, kh, vh, window=L), plain)
    np.testing.assert_array_equal(O.attend(q, kh, vh, window=10 * L), plain)
    # GQA equals repeated KV heads (group h // hpk)
    hpk = Hq // Hkv
    rep = O.attend(q, np.repeat(kh, hpk, axis=1), np.repeat(vh, hpk, axis=1))
    np.testing.assert_array_equal(rep, plain)
    # a wrong fan-out (h % Hkv) would differ
    wrong = O.attend(q, np.tile(kh, (1, hpk, 1)), np.tile(vh, (1, hpk, 1)))
    assert not np.allclose(wrong, plain)


def test_softcap_limits_and_saturation():
    """Score soft-capping (the softcap argument of cortiq-engine "Struct
    LayerKvCache" fn attend_group / attend_group_upto, read as the usual
    s -> c * tanh(s / c) on the scaled score, sink not capped), pinned by
    limits and a closed form rather than by restating it."""
    rng = np.random.default_rng(21)
    L, Hq, Hkv, D = 24, 4, 2, 32
    kh = rng.standard_normal((L, Hkv, D))
    vh = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((1, Hq, D))
    plain = O.attend(q, kh, vh)
    # a cap far above every score changes nothing (a missing "c *" or "/ c"
    # would make it uniform or explode)
    np.testing.assert_allclose(O.attend(q, kh, vh, softcap=1e9), plain, rtol=0, atol=1e-12)
    # softcap 0 is off
    np.testing.assert_array_equal(O.attend(q, kh, vh, softcap=0.0), plain)
    # saturation: huge scores cap to +-c exactly, so the weights are e^{+-c}
    # by sign of q.k alone; the sink (not capped) joins with e^{sink}
    c, sink = 1.5, 2.0
    qb = q * 1e6
    out = O.attend(qb, kh, vh, softcap=c, sinks=np.full(Hq, sink))
    hpk = Hq // Hkv
    for h in range(Hq):
        sgn = np.sign(kh[:, h // hpk, :] @ qb[0, h])
        w = np.exp(c * sgn)
        want = (w @ vh[:, h // hpk, :]) / (np.exp(sink) + w.sum())
        np.testing.assert_allclose(out[0, h], want, rtol=1e-12, atol=1e-12)


def test_causal_rows_equal_sequential_append_then_attend():
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D, T = 2, 8, 2, 64, 6
    prefix = rng.standard_normal((B, 20, Hkv, D)).astype(np.float32)
    kn = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    sinks = rng.standard_normal(Hq)
    for window in (0, 7):
        a = O.OracleKvCache(B, Hkv, D, window=window)
        a.append(prefix, prefix * 0.5)
        a.append(kn, vn)
        par = a.decode(q, sinks=sinks)
        s = O.OracleKvCache(B, Hkv, D, window=window)
        s.append(prefix, prefix * 0.5)
        for t in range(T):
            s.append(kn[:, t:t + 1], vn[:, t:t + 1])
            seq = s.decode(q[:, t:t + 1], sinks=sinks)
            np.testing.assert_array_equal(seq[:, 0], par[:, t])


def test_truncate_then_reappend_equals_clean_build():
    rng = np.random.default_rng(14)
    B, Hkv, D = 2, 2, 64
    k = rng.standard_normal((B, 30, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, 30, Hkv, D)).astype(np.float32)
    junk = rng.standard_normal((B, 8, Hkv, D)).astype(np.float32)
    a = O.OracleKvCache(B, Hkv, D)
    a.append(k[:, :20], v[:, :20])
    a.append(junk, junk)                        # a rejected draft
    a.truncate([20 + 3, 20 + 0])                # accept 3 and 0
    a.append(k[:1, 23:30], v[:1, 23:30], seq_ids=[0])
    a.append(k[1:, 20:30], v[1:, 20:30], seq_ids=[1])
    c = O.OracleKvCache(B, Hkv, D)
    kk = k.copy()
    vv = v.copy()
    kk[0, 20:23] = junk[0, :3]
    vv[0, 20:23] = junk[0, :3]
    c.append(kk, vv)
    for b in range(B):
        for x, y in zip(a.rows(b), c.rows(b)):
            np.testing.assert_array_equal(x, y)


def test_decode_window_suffix_shortcut():
    # decode() dequantises only rows some query can see; compare with the
    # plain attend() over all rows
    rng = np.random.default_rng(15)
    Hq, Hkv, D, L, T, W = 4, 2, 32, 50, 3, 9
    c = O.OracleKvCache(1, Hkv, D, window=W)
    c.append(rng.standard_normal((1, L, Hkv, D)).astype(np.float32),
             rng.standard_normal((1, L, Hkv, D)).astype(np.float32))
    q = rng.standard_normal((1, T, Hq, D))
    kr, vr = c.rows(0)
    full = O.attend(q[0], O.dequantize_k_rows(kr, Hkv, D), O.dequantize_v_rows(vr, Hkv, D), window=W)
    np.testing.assert_array_equal(c.decode(q)[0], full)


# ---------------------------------------------------------------- FP8 E4M3

def _torch_e4m3_table():
    """float64 value of every E4M3 byte by torch's float8_e4m3fn decoding."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_known_encodings():
    with open(os.path.join(GOLD, "e4m3_known.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    vals = np.array([_parse_float(r[0]) for r in rows])
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    np.testing.assert_array_equal(O.e4m3_bits(vals), want)


def test_e4m3_decode_every_byte_matches_torch():
    want = _torch_e4m3_table()
    got = O.e4m3_value(np.arange(256))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    np.testing.assert_array_equal(got[fin], want[fin])
    np.testing.assert_array_equal(np.signbit(got[fin]), np.signbit(want[fin]))
    assert np.nanmax(got) == O.E4M3_MAX and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_e4m3_encode_is_nearest_finite_code_ties_even():
    """Brute force: the byte of |y| is the finite non-negative code whose
    torch-decoded value is nearest (ties to the even code), the sign bit that
    of y; this also covers saturation beyond 448."""
    table = _torch_e4m3_table()
    grid = table[:0x7F]                                  # bytes 0x00..0x7E, increasing
    rng = np.random.default_rng(21)
    y = [np.ldexp(rng.uniform(1.0, 2.0, 40000), rng.integers(-13, 11, 40000))
         * rng.choice([-1.0, 1.0], 40000)]
    mids = (grid[1:] + grid[:-1]) / 2                    # every tie
    y += [mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf)]
    y += [np.array([0.0, -0.0, 447.9, 448.0, 463.9, 464.0, 464.1, 500.0, 1e30, -1e30])]
    y = np.concatenate(y)
    # beyond 1000 every finite code is farther than 448; clipping there keeps
    # the distances exact in float64
    a = np.minimum(np.abs(y), 1000.0)
    dist = np.abs(a[:, None] - grid[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    n_cand = cand.sum(axis=1)
    assert n_cand.max() <= 2
    first = np.argmax(cand, axis=1)
    pick = np.where((n_cand == 2) & (first % 2 == 1), first + 1, first)
    want = (pick | (np.signbit(y).astype(np.int64) << 7)).astype(np.uint8)
    np.testing.assert_array_equal(O.e4m3_bits(y), want)


def test_e4m3_encode_matches_torch_in_range():
    """torch's float -> float8_e4m3fn cast (round to nearest even) on float32
    values below the 464 tie, above which torch gives NaN and the format here
    saturates."""
    rng = np.random.default_rng(22)
    x = np.concatenate([rng.standard_normal(200000), 30 * rng.standard_normal(200000),
                        np.ldexp(rng.uniform(-2, 2, 200000), rng.integers(-12, 0, 200000))])
    x = x[np.abs(x) < 464].astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_bits(x.astype(np.float64)), want)


def test_e4m3_round_trip_and_error_bound():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(O.e4m3_bits(O.e4m3_value(codes)), codes.astype(np.uint8))
    rng = np.random.default_rng(23)
    x = rng.uniform(-448, 448, 100000) * np.ldexp(1.0, rng.integers(-14, 1, 100000))
    err = np.abs(x - O.e4m3_value(O.e4m3_bits(x)))
    # half the spacing of the binade: 2^(max(floor(log2|x|), -6) - 4)
    e = np.maximum(np.floor(np.log2(np.abs(x))), -6)
    assert np.all(err <= np.ldexp(1.0, (e - 4).astype(int)))
    with pytest.raises(ValueError):
        O.e4m3_bits(np.array([np.inf]))


def test_e4m3_cache_rows_and_attention_on_representable_values():
    """With inputs that E4M3 holds exactly, the e4m3 cache stores each row as
    its elements' bytes in [token, kv_head, dim] order and its decode equals
    torch SDPA on the raw inputs."""
    rng = np.random.default_rng(24)
    table = _torch_e4m3_table()
    fin = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    n_seq, L, Hkv, D, Hq, T = 2, 40, 2, 64, 8, 3
    kc = rng.choice(fin[np.abs(table[fin]) <= 4], (n_seq, L, Hkv, D))
    vc = rng.choice(fin, (n_seq, L, Hkv, D))
    k, v = table[kc].astype(np.float32), table[vc].astype(np.float32)
    c = O.OracleKvCache(n_seq, Hkv, D, fmt="e4m3")
    assert c.k_tok == c.v_tok == Hkv * D
    c.append(k[:, :25], v[:, :25])
    c.append(k[:, 25:], v[:, 25:])
    for b in range(n_seq):
        kr, vr = c.rows(b)
        np.testing.assert_array_equal(kr, kc[b].reshape(L, -1).astype(np.uint8))
        np.testing.assert_array_equal(vr, vc[b].reshape(L, -1).astype(np.uint8))
    q = rng.standard_normal((n_seq, T, Hq, D)) * 0.1
    sinks = rng.standard_normal(Hq)
    got = c.decode(q, sinks=sinks)
    for b in range(n_seq):
        ref = _sdpa_reference(q[b], k[b].astype(np.float64), v[b].astype(np.float64),
                              scale=1 / math.sqrt(D), sinks=sinks, window=0)
        np.testing.assert_allclose(got[b], ref, rtol=1e-11, atol=1e-11)


def test_rollback_by_accept_count_equals_clean_build():
    """After a T-row draft step, rollback(accept) leaves exactly the bytes of a
    cache built from the snapshot rows plus the first accept draft rows."""
    rng = np.random.default_rng(31)
    n_kv, D, T = 2, 64, 6
    snap = rng.standard_normal((2, 9, n_kv, D)).astype(np.float32)
    draft = rng.standard_normal((2, T, n_kv, D)).astype(np.float32)
    for fmt in ("q8_0/q5_1", "e4m3"):
        c = O.OracleKvCache(2, n_kv, D, fmt=fmt)
        c.append(snap, snap)
        c.append(draft, -draft)
        c.rollback([0, 4], T)
        assert c.lens() == [9, 13]
        clean = O.OracleKvCache(2, n_kv, D, fmt=fmt)
        clean.append(snap, snap)
        clean.append(draft[:, :4], -draft[:, :4], )
        clean.truncate([9, 13])
        for b in range(2):
            for x, y in zip(c.rows(b), clean.rows(b)):
                np.testing.assert_array_equal(x, y)
        with pytest.raises(ValueError):
            c.rollback([T + 1, 0], T)
        with pytest.raises(ValueError):
            c.rollback([-1, 0], T)
