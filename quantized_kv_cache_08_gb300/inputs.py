"""Seeded synthetic inputs for the five decode workloads.

This module holds only random-number plumbing and workload shapes; none of
the cache's arithmetic.  The tests, the smoke entry point and the benchmark
draw from it, and feed the same host arrays to the CUDA path and to the CPU
oracle.  Every tensor is produced on the CPU by a torch.Generator seeded from
(workload seed, sequence, 1024-row chunk, stream), so any row range of any
sequence can be regenerated on its own, in any order.

Workloads (no dataset is involved; these stand in for the decode shapes the
pages describe):
  ctx512      1 sequence, 8 Q / 2 KV heads, head_dim 128, 512 rows, T=1
  ctx32k      1 sequence, 32 Q / 8 KV heads, head_dim 128, 32768 rows, T=1,
              q in bf16, 1% of the K and V channels scaled by 10
  batch64     64 sequences, 32 Q / 8 KV heads, head_dim 128, lengths uniform
              in [1024, 16384] at decode (prefill len-1, a 64-row append),
              T=1
  swa_ring    1 sequence, 64 Q / 8 KV heads, head_dim 64, a sink logit per Q
              head ~ N(0,1), window 4096 over a ring of window+31 rows,
              T=1 steps until the length reaches 131072
  spec_verify 1 sequence, 16 Q / 4 KV heads, head_dim 256, 16384 rows, then
              100 rounds of: append T=8, decode T=8 causal, keep
              accept ~ U{0..8} of the 8 rows
K, V and q are N(0,1) float32 unless stated.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

CHUNK = 1024

WORKLOADS = {
    "ctx512": dict(index=1, n_seq=1, n_q=8, n_kv=2, head_dim=128, ctx=512, T=1,
                   q_dtype="f32", outlier_frac=0.0, window=0, ring=False, sinks=False),
    "ctx32k": dict(index=2, n_seq=1, n_q=32, n_kv=8, head_dim=128, ctx=32768, T=1,
                   q_dtype="bf16", outlier_frac=0.01, window=0, ring=False, sinks=False),
    "batch64": dict(index=3, n_seq=64, n_q=32, n_kv=8, head_dim=128, ctx=(1024, 16384), T=1,
                    q_dtype="f32", outlier_frac=0.0, window=0, ring=False, sinks=False),
    "swa_ring": dict(index=4, n_seq=1, n_q=64, n_kv=8, head_dim=64, ctx=131072, T=1,
                     q_dtype="f32", outlier_frac=0.0, window=4096, ring=True, sinks=True),
    "spec_verify": dict(index=5, n_seq=1, n_q=16, n_kv=4, head_dim=256, ctx=16384, T=8,
                        q_dtype="f32", outlier_frac=0.0, window=0, ring=False, sinks=False,
                        rounds=100),
}

BASE_SEED = 20261202


def _gen(*key) -> torch.Generator:
    s = BASE_SEED
    for k in key:
        s = (s * 1000003 + int(k) + 1) % (2 ** 62)
    g = torch.Generator()
    g.manual_seed(s)
    return g


@dataclass
class Workload:
    name: str
    index: int
    n_seq: int
    n_q: int
    n_kv: int
    head_dim: int
    T: int
    q_dtype: str
    window: int
    ring: bool
    sinks: bool
    outlier_frac: float
    ctx: object
    rounds: int = 0
    _outliers: dict = field(default_factory=dict)

    @property
    def kvd(self):
        return self.n_kv * self.head_dim

    # ---- per-workload draws
    def lengths(self):
        """Per-sequence length at decode time."""
        if isinstance(self.ctx, tuple):
            lo, hi = self.ctx
            return torch.randint(lo, hi + 1, (self.n_seq,), generator=_gen(self.index, 1)).tolist()
        return [int(self.ctx)] * self.n_seq

    def accepts(self):
        """accept_len of each verify round, uniform in 0..T."""
        return torch.randint(0, self.T + 1, (self.rounds,), generator=_gen(self.index, 2)).tolist()

    def sink_logits(self):
        if not self.sinks:
            return None
        return torch.randn(self.n_q, generator=_gen(self.index, 3), dtype=torch.float32)

    def outlier_channels(self, which):
        """Channel indices (of kvd) scaled by 10 in K (which=0) or V (which=1)."""
        if which not in self._outliers:
            n = int(round(self.outlier_frac * self.kvd))
            perm = torch.randperm(self.kvd, generator=_gen(self.index, 4, which))
            self._outliers[which] = perm[:n].sort().values
        return self._outliers[which]

    # ---- rows
    def _chunk(self, seq, chunk, which):
        g = _gen(self.index, 10 + which, seq, chunk)
        x = torch.randn(CHUNK, self.kvd, generator=g, dtype=torch.float32)
        ch = self.outlier_channels(which)
        if len(ch):
            x[:, ch] *= 10.0
        return x

    def rows(self, seq, lo, hi, which):
        """float32 [hi-lo, n_kv, head_dim] of K (which=0) or V (which=1)."""
        parts = []
        for c in range(lo // CHUNK, (hi + CHUNK - 1) // CHUNK):
            x = self._chunk(seq, c, which)
            a = max(lo, c * CHUNK) - c * CHUNK
            b = min(hi, (c + 1) * CHUNK) - c * CHUNK
            parts.append(x[a:b])
        if not parts:
            return torch.zeros(0, self.n_kv, self.head_dim)
        return torch.cat(parts).view(hi - lo, self.n_kv, self.head_dim)

    def kv(self, seq, lo, hi):
        return self.rows(seq, lo, hi, 0), self.rows(seq, lo, hi, 1)

    def q(self, step, T=None):
        """q of decode step `step`: [n_seq, T, n_q, head_dim], float32 or bf16."""
        T = self.T if T is None else T
        x = torch.randn(self.n_seq, T, self.n_q, self.head_dim, generator=_gen(self.index, 5, step),
                        dtype=torch.float32)
        if self.q_dtype == "bf16":
            x = x.to(torch.bfloat16)
        return x


def workload(name, **override) -> Workload:
    spec = dict(WORKLOADS[name])
    spec.update(override)
    return Workload(name=name, **spec)
