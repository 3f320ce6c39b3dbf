"""kvq oracle: a plain, slow fp64 CPU statement of the quantised KV cache.

TEST INFRASTRUCTURE.  Only the test-suite, the package's smoke entry point and
the CPU-baseline leg of the benchmark may import this module.  The product path
(the CUDA library and its Python binding) never imports it and has no CPU
fallback.  This module shares no code, table or constant generator with the
CUDA path; it takes plain numpy arrays in and gives numpy arrays out.

What it states, and which passage each piece follows
----------------------------------------------------
* Block formats (memra-engine "Struct KvLayer", type description; and the
  KvLayer entry of "Module cache"): K is stored q8_0, 34 bytes per 32 elements;
  V is stored q5_1, 24 bytes per 32 elements.  The field contents are read as:
    q8_0: fp16 scale d = amax/127 (round-to-nearest-even), then 32 int8 codes
          c = round-half-away-from-zero(x/d), clamped to [-127, 127].
    q5_1: fp16 d = (max-min)/31, fp16 m = min, a little-endian u32 `qh` whose
          bit i is bit 4 of code i, then 16 bytes `qs` where byte j holds the
          low nibble of code j (bits 0-3) and of code j+16 (bits 4-7); codes
          u = round-half-away((x-m)/d) clamped to [0, 31], taken against the
          STORED (fp16-rounded) m and d.
  fp16 here is IEEE 754 binary16, written out below from its definition.
* Row placement ("Struct KvLayer", type description): a token row keeps the
  [token, kv_head, dim] order; element index e = kv_head*head_dim + d goes to
  block e // 32, lane e % 32; a block never straddles a head (head_dim % 32 == 0).
* Attention (cortiq-engine "Struct LayerKvCache"):
    - GQA fan-out: Q head h reads KV group h // hpk (fn o1_views);
    - score scale 1/sqrt(head_dim) unless overridden (fn attend_group);
    - sliding window: rows before first = stored - window get probability 0
      (fn attend_group and fn attend_group_upto);
    - T query rows: row i sees the first upto = s0 + i + 1 stored rows
      (fn attend_group_upto);
    - learned sink: one logit per Q head, joins the softmax max and adds
      exp(sink - max) to the denominator, carries no value (field sinks,
      fn attend_group_upto).
* Rollback ("Struct Cache", fn rollback, item C.1): len = snapshot_len +
  accept_len, truncate without copy; cortiq-engine fn truncate_last.

The logical cache model here is flat: every sequence is a list of all rows it
holds, with no ring.  A ring on the device is a re-addressing of these rows
(memra-engine "Struct KvLayer", fields ring and base_d), so its live bytes
must equal the logical rows of this model.

All arithmetic is float64.  numpy vectorises over independent blocks, rows and
heads only; there is no blocking, fusion or reordering beyond the formulas.
"""

from __future__ import annotations

import math

import numpy as np

QK = 32                 # elements per block
Q8_0_BYTES = 34         # 2 (fp16 d) + 32 (int8 codes)
Q5_1_BYTES = 24         # 2 (fp16 d) + 2 (fp16 m) + 4 (qh) + 16 (qs)


# ---------------------------------------------------------------------------
# IEEE 754 binary16 (1 sign bit, 5 exponent bits with bias 15, 10 fraction
# bits).  Normal numbers are (1 + f/1024) * 2**(E-15) for E in 1..30;
# subnormals are f * 2**-24; E = 31 encodes infinity.
# ---------------------------------------------------------------------------

def f16_bits(y) -> np.ndarray:
    """Encode float64 values as binary16 bit patterns, rounding to nearest,
    ties to even.  Values whose rounded magnitude exceeds 65504 become inf.
    Raises on NaN/inf input."""
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        raise ValueError("f16_bits: non-finite input")
    sign = np.signbit(y).astype(np.uint32)
    a = np.abs(y)
    _, ex = np.frexp(a)                   # a = m * 2**ex, m in [0.5, 1); exact
    e = np.maximum(ex.astype(np.int64) - 1, -14)   # binade; below 2**-14 the
    quantum = np.ldexp(1.0, e - 10)                # subnormal step 2**-24 holds
    n = a / quantum                       # exact: a power-of-two divisor
    r = np.rint(n)                        # nearest integer, ties to even
    r = r.astype(np.int64)
    carry = r == 2048                     # rounded up into the next binade
    e = np.where(carry, e + 1, e)
    r = np.where(carry, 1024, r)
    sub = r < 1024                        # only possible when e == -14
    biased = np.where(sub, 0, e + 15)
    frac = np.where(sub, r, r - 1024)
    over = biased >= 31
    biased = np.where(over, 31, biased)
    frac = np.where(over, 0, frac)
    bits = (sign << 15) | (biased.astype(np.uint32) << 10) | frac.astype(np.uint32)
    return bits.astype(np.uint16)


def f16_value(bits) -> np.ndarray:
    """Decode binary16 bit patterns to float64 (exact).  NaN patterns -> nan."""
    b = np.asarray(bits).astype(np.int64)
    s = np.where((b >> 15) & 1, -1.0, 1.0)
    E = (b >> 10) & 31
    f = b & 1023
    mag = np.where(E == 0, np.ldexp(f.astype(np.float64), -24),
                   np.ldexp((1024 + f).astype(np.float64), (E - 25).astype(np.int64)))
    mag = np.where(E == 31, np.where(f == 0, np.inf, np.nan), mag)
    return s * mag


def round_half_away(t) -> np.ndarray:
    """sign(t) * (nearest integer to |t|, halves going away from zero).
    Exact for every float64 t: the fraction |t| - floor(|t|) is exact."""
    t = np.asarray(t, dtype=np.float64)
    a = np.abs(t)
    fl = np.floor(a)
    n = fl + (a - fl >= 0.5)
    return np.copysign(n, t)


# ---------------------------------------------------------------------------
# q8_0 (K plane)
# ---------------------------------------------------------------------------

def q8_0_quantize(x) -> np.ndarray:
    """Quantise float32 blocks [..., 32] to q8_0 bytes [..., 34].

    d = fp16(amax / 127); c_i = clamp(round_half_away(x_i / d), -127, 127)
    with d the stored fp16 value; all codes are 0 when d rounds to 0.
    Layout: d as little-endian fp16, then c_0..c_31 as int8."""
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] != QK:
        raise ValueError("q8_0_quantize: last axis must be 32")
    x = x.astype(np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("q8_0_quantize: non-finite input")
    amax = np.max(np.abs(x), axis=-1)
    d_bits = f16_bits(amax / 127.0)
    d = f16_value(d_bits)
    if not np.all(np.isfinite(d)):
        raise ValueError("q8_0_quantize: scale overflows fp16")
    dd = d[..., None]
    safe = np.where(dd == 0, 1.0, dd)
    c = np.where(dd == 0, 0.0, np.clip(round_half_away(x / safe), -127, 127))
    out = np.empty(x.shape[:-1] + (Q8_0_BYTES,), dtype=np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2:] = c.astype(np.int8).view(np.uint8)
    return out


def q8_0_fields(blk):
    """Split q8_0 bytes [..., 34] into (d float64 [...], codes int [..., 32])."""
    blk = np.asarray(blk, dtype=np.uint8)
    d_bits = blk[..., 0].astype(np.uint16) | (blk[..., 1].astype(np.uint16) << 8)
    codes = blk[..., 2:].view(np.int8).astype(np.int64)
    return f16_value(d_bits), codes


def q8_0_dequantize(blk) -> np.ndarray:
    """q8_0 bytes [..., 34] -> float64 [..., 32]: x_hat = d * c (exact)."""
    d, c = q8_0_fields(blk)
    return d[..., None] * c


# ---------------------------------------------------------------------------
# q5_1 (V plane)
# ---------------------------------------------------------------------------

def q5_1_quantize(x) -> np.ndarray:
    """Quantise float32 blocks [..., 32] to q5_1 bytes [..., 24].

    d = fp16((max - min)/31), m = fp16(min);
    u_i = clamp(round_half_away((x_i - m)/d), 0, 31) with the stored m and d;
    all codes 0 when d rounds to 0.
    Layout: d (fp16 LE), m (fp16 LE), qh (u32 LE, bit i = bit 4 of u_i),
    qs[j] = (u_j & 15) | ((u_{j+16} & 15) << 4) for j = 0..15."""
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] != QK:
        raise ValueError("q5_1_quantize: last axis must be 32")
    x = x.astype(np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("q5_1_quantize: non-finite input")
    mn = np.min(x, axis=-1)
    mx = np.max(x, axis=-1)
    d_bits = f16_bits((mx - mn) / 31.0)
    m_bits = f16_bits(mn)
    d = f16_value(d_bits)
    m = f16_value(m_bits)
    if not (np.all(np.isfinite(d)) and np.all(np.isfinite(m))):
        raise ValueError("q5_1_quantize: scale or min overflows fp16")
    dd = d[..., None]
    safe = np.where(dd == 0, 1.0, dd)
    u = np.where(dd == 0, 0.0,
                 np.clip(round_half_away((x - m[..., None]) / safe), 0, 31))
    u = u.astype(np.uint32)
    qh = np.zeros(x.shape[:-1], dtype=np.uint32)
    for i in range(QK):
        qh |= ((u[..., i] >> 4) & 1) << np.uint32(i)
    qs = (u[..., :16] & 15) | ((u[..., 16:] & 15) << 4)
    out = np.empty(x.shape[:-1] + (Q5_1_BYTES,), dtype=np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2] = (m_bits & 0xFF).astype(np.uint8)
    out[..., 3] = (m_bits >> 8).astype(np.uint8)
    for k in range(4):
        out[..., 4 + k] = ((qh >> np.uint32(8 * k)) & 0xFF).astype(np.uint8)
    out[..., 8:] = qs.astype(np.uint8)
    return out


def q5_1_fields(blk):
    """Split q5_1 bytes [..., 24] into (d, m float64 [...], u int [..., 32])."""
    blk = np.asarray(blk, dtype=np.uint8)
    d_bits = blk[..., 0].astype(np.uint16) | (blk[..., 1].astype(np.uint16) << 8)
    m_bits = blk[..., 2].astype(np.uint16) | (blk[..., 3].astype(np.uint16) << 8)
    qh = np.zeros(blk.shape[:-1], dtype=np.int64)
    for k in range(4):
        qh |= blk[..., 4 + k].astype(np.int64) << (8 * k)
    qs = blk[..., 8:].astype(np.int64)
    u = np.empty(blk.shape[:-1] + (QK,), dtype=np.int64)
    for j in range(16):
        u[..., j] = (qs[..., j] & 15) | (((qh >> j) & 1) << 4)
        u[..., j + 16] = (qs[..., j] >> 4) | (((qh >> (j + 16)) & 1) << 4)
    return f16_value(d_bits), f16_value(m_bits), u


def q5_1_dequantize(blk) -> np.ndarray:
    """q5_1 bytes [..., 24] -> float64 [..., 32]: x_hat = d*u + m (exact)."""
    d, m, u = q5_1_fields(blk)
    return d[..., None] * u + m[..., None]


# ---------------------------------------------------------------------------
# FP8 E4M3 (the alternative K/V format: one byte per element, no block scale)
#
# memra-engine "Module cache", items KV_FP8_FORCE, gkv_on (the FP8-GLOBALS
# switch) and kv_fp8_on: K and V are held as e4m3 ("kf8vf8").  The pages name the format
# only; it is read as OCP FP8 E4M3: 1 sign bit, 4 exponent bits with bias 7,
# 3 fraction bits, no infinities.  Normals are (1 + f/8) * 2**(E-7) for
# E in 1..15 except E = 15, f = 7 (NaN); subnormals are f/8 * 2**-6; the
# largest finite magnitude is 1.75 * 2**8 = 448.  Each element is encoded on
# its own, with no scale: round to nearest, ties to even, and magnitudes
# above 448 saturate to 448 (there is no infinity to overflow to).
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_bits(y) -> np.ndarray:
    """Encode finite float64 values as E4M3 bytes (nearest, ties to even,
    saturating at +-448).  Raises on non-finite input."""
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        raise ValueError("e4m3_bits: non-finite input")
    sign = np.signbit(y).astype(np.int64)
    a = np.abs(y)
    _, ex = np.frexp(a)                   # a = m * 2**ex, m in [0.5, 1); exact
    e = np.maximum(ex.astype(np.int64) - 1, -6)    # binade; below 2**-6 the
    quantum = np.ldexp(1.0, e - 3)                 # subnormal step 2**-9 holds
    r = np.rint(a / quantum).astype(np.int64)      # ties to even; exact divisor
    carry = r == 16                       # rounded up into the next binade
    e = np.where(carry, e + 1, e)
    r = np.where(carry, 8, r)
    sub = r < 8                           # only possible when e == -6
    biased = np.where(sub, 0, e + 7)
    frac = np.where(sub, r, r - 8)
    over = (biased > 15) | ((biased == 15) & (frac == 7))
    biased = np.where(over, 15, biased)   # saturate to 448 = (1 + 6/8) * 2**8
    frac = np.where(over, 6, frac)
    return ((sign << 7) | (biased << 3) | frac).astype(np.uint8)


def e4m3_value(bits) -> np.ndarray:
    """Decode E4M3 bytes to float64 (exact).  0x7F and 0xFF are NaN."""
    b = np.asarray(bits).astype(np.int64)
    s = np.where((b >> 7) & 1, -1.0, 1.0)
    E = (b >> 3) & 15
    f = b & 7
    mag = np.where(E == 0, np.ldexp(f.astype(np.float64), -9),
                   np.ldexp((8 + f).astype(np.float64), (E - 10).astype(np.int64)))
    mag = np.where((E == 15) & (f == 7), np.nan, mag)
    return s * mag


# ---------------------------------------------------------------------------
# Token rows: [token, kv_head, dim] element order, 32-element blocks
# ---------------------------------------------------------------------------

def _blocks_of_rows(x, n_kv, head_dim):
    x = np.asarray(x, dtype=np.float32)
    if head_dim % QK:
        raise ValueError("head_dim must be a multiple of 32")
    kvd = n_kv * head_dim
    flat = x.reshape(-1, kvd)          # element e = kv_head*head_dim + d
    return flat.reshape(-1, kvd // QK, QK)   # block e // 32, lane e % 32


def quantize_k_rows(k, n_kv, head_dim) -> np.ndarray:
    """K rows [..., n_kv, head_dim] float32 -> [n_rows, kb*34] uint8."""
    blocks = _blocks_of_rows(k, n_kv, head_dim)
    return q8_0_quantize(blocks).reshape(blocks.shape[0], -1)


def quantize_v_rows(v, n_kv, head_dim) -> np.ndarray:
    """V rows [..., n_kv, head_dim] float32 -> [n_rows, kb*24] uint8."""
    blocks = _blocks_of_rows(v, n_kv, head_dim)
    return q5_1_quantize(blocks).reshape(blocks.shape[0], -1)


def e4m3_rows(x, n_kv, head_dim) -> np.ndarray:
    """K or V rows [..., n_kv, head_dim] float32 -> [n_rows, n_kv*head_dim]
    E4M3 bytes, element e = kv_head*head_dim + d at byte e of its row."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1, n_kv * head_dim).astype(np.float64)
    return e4m3_bits(flat)


def dequantize_e4m3_rows(rows, n_kv, head_dim) -> np.ndarray:
    """[n_rows, n_kv*head_dim] E4M3 bytes -> float64 [n_rows, n_kv, head_dim]."""
    rows = np.asarray(rows, dtype=np.uint8)
    return e4m3_value(rows).reshape(rows.shape[0], n_kv, head_dim)


def dequantize_k_rows(rows, n_kv, head_dim) -> np.ndarray:
    """[n_rows, kb*34] -> float64 [n_rows, n_kv, head_dim]."""
    rows = np.asarray(rows, dtype=np.uint8)
    blk = rows.reshape(rows.shape[0], -1, Q8_0_BYTES)
    return q8_0_dequantize(blk).reshape(rows.shape[0], n_kv, head_dim)


def dequantize_v_rows(rows, n_kv, head_dim) -> np.ndarray:
    """[n_rows, kb*24] -> float64 [n_rows, n_kv, head_dim]."""
    rows = np.asarray(rows, dtype=np.uint8)
    blk = rows.reshape(rows.shape[0], -1, Q5_1_BYTES)
    return q5_1_dequantize(blk).reshape(rows.shape[0], n_kv, head_dim)


# ---------------------------------------------------------------------------
# Attention over one sequence's dequantised rows
# ---------------------------------------------------------------------------

def attend(q, k_hat, v_hat, *, scale=None, sinks=None, window=0,
           heads=None, rows_t=None, softcap=0.0):
    """Decode attention of the last T rows of one sequence.

    q      [T, Hq, D]  (any float dtype; taken exactly as float64)
    k_hat  [L, Hkv, D] float64 dequantised keys, logical rows 0..L-1
    v_hat  [L, Hkv, D] float64 dequantised values
    Query row t sits at position s0 + t (s0 = L - T) and sees rows
    [lstart_t, upto_t) with upto_t = s0 + t + 1 and lstart_t =
    max(0, upto_t - window) when window > 0, else 0.
    Head h reads KV group h // (Hq // Hkv).  Scores are scale * <q, k_hat>,
    scale = 1/sqrt(D) when None.  A sink logit (per Q head, not scaled) joins
    the max and the denominator and carries no value.
    softcap > 0 caps every scaled score s to softcap * tanh(s / softcap) before
    the softmax (the pages pass a softcap to fn attend_group / attend_group_upto
    without defining it; this is the usual logit soft-capping); the sink logit
    is not capped.
    `heads` / `rows_t` restrict the computation to a subset (others are nan).
    Returns float64 [T, Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    L, Hkv, _ = k_hat.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if T > L:
        raise ValueError("fewer stored rows than query rows")
    hpk = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    s0 = L - T
    out = np.full((T, Hq, D), np.nan)
    for t in (range(T) if rows_t is None else rows_t):
        upto = s0 + t + 1
        lstart = max(0, upto - window) if window > 0 else 0
        for h in (range(Hq) if heads is None else heads):
            g = h // hpk
            kk = k_hat[lstart:upto, g, :]
            vv = v_hat[lstart:upto, g, :]
            s = scale * (kk @ q[t, h])
            if softcap > 0:
                s = softcap * np.tanh(s / softcap)
            sink = -math.inf if sinks is None else float(sinks[h])
            mx = max(sink, float(np.max(s)))
            w = np.exp(s - mx)
            denom = math.exp(sink - mx) + float(np.sum(w))
            out[t, h] = (w @ vv) / denom
    return out


# ---------------------------------------------------------------------------
# Logical cache model
# ---------------------------------------------------------------------------

class OracleKvCache:
    """Flat logical model of a layer cache holding n_seq sequences.

    append() quantises rows exactly as the formats above state and places them
    at row `len` of each target sequence; truncate() drops rows past the new
    length (rollback: len = snapshot_len + accept_len, no copy); decode()
    attends the last T rows of every sequence over its dequantised rows.
    fmt "q8_0/q5_1" stores K as q8_0 and V as q5_1 blocks; fmt "e4m3" stores
    both as one E4M3 byte per element."""

    def __init__(self, n_seq, n_kv, head_dim, window=0, fmt="q8_0/q5_1"):
        if head_dim % QK:
            raise ValueError("head_dim must be a multiple of 32")
        if fmt not in ("q8_0/q5_1", "e4m3"):
            raise ValueError("fmt must be 'q8_0/q5_1' or 'e4m3'")
        self.n_seq, self.n_kv, self.head_dim, self.window = n_seq, n_kv, head_dim, window
        self.fmt = fmt
        self.kb = n_kv * head_dim // QK
        if fmt == "e4m3":
            self.k_tok = self.v_tok = n_kv * head_dim
        else:
            self.k_tok = self.kb * Q8_0_BYTES
            self.v_tok = self.kb * Q5_1_BYTES
        self._k = [np.zeros((0, self.k_tok), np.uint8) for _ in range(n_seq)]
        self._v = [np.zeros((0, self.v_tok), np.uint8) for _ in range(n_seq)]

    def lens(self):
        return [r.shape[0] for r in self._k]

    def append(self, k, v, seq_ids=None):
        """k, v: [n, T, n_kv, head_dim] float32; row t of entry i goes to
        sequence seq_ids[i] (all sequences in order when None)."""
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        ids = list(range(self.n_seq)) if seq_ids is None else list(seq_ids)
        if k.shape[0] != len(ids) or v.shape != k.shape:
            raise ValueError("append: shape mismatch")
        for i, b in enumerate(ids):
            if self.fmt == "e4m3":
                kr = e4m3_rows(k[i], self.n_kv, self.head_dim)
                vr = e4m3_rows(v[i], self.n_kv, self.head_dim)
            else:
                kr = quantize_k_rows(k[i], self.n_kv, self.head_dim)
                vr = quantize_v_rows(v[i], self.n_kv, self.head_dim)
            self._k[b] = np.concatenate([self._k[b], kr])
            self._v[b] = np.concatenate([self._v[b], vr])

    def append_bytes(self, b, k_rows, v_rows):
        """Place already-quantised rows (used to feed identical bytes)."""
        self._k[b] = np.concatenate([self._k[b], np.asarray(k_rows, np.uint8)])
        self._v[b] = np.concatenate([self._v[b], np.asarray(v_rows, np.uint8)])

    def truncate(self, new_len):
        for b, n in enumerate(new_len):
            if n < 0 or n > self._k[b].shape[0]:
                raise ValueError("truncate: length out of range")
            self._k[b] = self._k[b][:n]
            self._v[b] = self._v[b][:n]

    def rollback(self, accept, T):
        """Rollback after a T-row draft step ("Struct Cache", fn rollback,
        item C.1): len = snapshot_len + accept_len with snapshot_len = len - T,
        so the first accept[b] of each sequence's last T rows stay."""
        lens = self.lens()
        new = []
        for b, a in enumerate(accept):
            a = int(a)
            if not 0 <= a <= T or lens[b] < T:
                raise ValueError("rollback: accept out of range")
            new.append(lens[b] - T + a)
        self.truncate(new)

    def rows(self, b, lo=0, hi=None):
        """Quantised bytes of logical rows [lo, hi) of sequence b."""
        return self._k[b][lo:hi], self._v[b][lo:hi]

    def decode(self, q, *, scale=None, sinks=None, heads=None, rows_t=None,
               seqs=None, softcap=0.0):
        """q [B, T, Hq, D] -> float64 [B, T, Hq, D] (nan where not computed)."""
        q = np.asarray(q, dtype=np.float64)
        out = np.full(q.shape, np.nan)
        for b in (range(self.n_seq) if seqs is None else seqs):
            L = self._k[b].shape[0]
            T = q.shape[1]
            lo = 0
            if self.window > 0:
                lo = max(0, L - T + 1 - self.window)   # rows no query row sees
            if self.fmt == "e4m3":
                kh = dequantize_e4m3_rows(self._k[b][lo:], self.n_kv, self.head_dim)
                vh = dequantize_e4m3_rows(self._v[b][lo:], self.n_kv, self.head_dim)
            else:
                kh = dequantize_k_rows(self._k[b][lo:], self.n_kv, self.head_dim)
                vh = dequantize_v_rows(self._v[b][lo:], self.n_kv, self.head_dim)
            # rows before `lo` have probability exactly 0 for every query row,
            # so attending the suffix with the same window is the same result
            out[b] = attend(q[b], kh, vh, scale=scale, sinks=sinks,
                            window=self.window, heads=heads, rows_t=rows_t,
                            softcap=softcap)
        return out
