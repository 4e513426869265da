"""Seeded synthetic workloads for the DropKV scoring path.

This module only builds inputs: query windows, K/V caches, sequence lengths and
eviction counts. It computes none of the method (no softmax, no scores, no
selection), so both the CUDA path and the CPU oracle can be fed from it.

The pages measure on real models over RULER and LongBench; those suites and
weights are not used here. These workloads stand in for them with the layer
shapes the pages name (Llama-3.1-8B-like GQA 32/8 with d=128, a Phi-3-mini-like
MHA layer, a Qwen-like batched ragged layer, w=8 tail queries, 5% and 10%
budgets, n up to 128K; "DropKV: Decoupling Residual-Output Perturbation ...",
Section 5 and Figure 3 caption).

Recipe (numpy PCG64, one generator per workload, fixed draw order):
  lengths (ragged workloads only) -> Q -> K -> V -> per KV head: outlier
  channels, their scales -> per KV head: sink -> per KV head: needles.
* Q, K, V: i.i.d. N(0, 1) float32.
* Outliers: 4 channels per KV head, shared by the keys of that head and the
  queries of its GQA group, with a scale s ~ exp(U[ln 2, ln 8]) per channel.
  The channel's term of every logit q.k is scaled by s (both the query and the
  key channel are multiplied by sqrt(s)).
* Attention sink: key 0 of each KV head is replaced by the minimum-norm vector
  whose logit with every window row r equals ln(n_b) + sigma_r^2 / 2 (the
  typical log-sum-exp of the other keys; sigma_r^2 = sum_c q_rc^2 s_c / d is the
  variance of row r's logit against an i.i.d. key), so each row puts roughly
  half its mass on the sink.  This is a least-squares solve on the queries.
* Needles: 64 keys per KV head at positions drawn without replacement from
  [1, n_b - w), each aligned with one window query q_r of the group (r drawn
  uniformly): key j becomes |k_j| (0.8 q_r/|q_r| + 0.6 w_j), w_j a random unit
  vector orthogonal to q_r (cosine 0.8 with that query).
* Sink mass (optional, `sink_margin` nats): the sink's target logit is raised
  by the margin, so each row puts roughly p0 = 1 / (1 + exp(-margin)) of its
  mass on the sink (margin = ln(p0 / (1 - p0))); 0 keeps the half-mass sink.
* Value offset (optional, `v_offset` = sigma): after the needles, every KV
  head draws a per-channel mean mu_c ~ N(0, sigma^2) plus 4 value outlier
  channels with mu_c = +-4 sigma, added to all of its values (V = mu + N(0, 1)),
  the common offset real value caches carry; |v|^2 is then far above
  |a - v|^2.
* Everything is rounded to bf16 (round to nearest even) once; the GPU and the
  oracle see exactly those bf16 values.  The tiny workload also keeps its
  float32 draws for the oracle's own self-checks.
* Eviction count per sequence: k_b = floor((100 - P) * (n_b - w) / 100) for a
  kept budget of P percent (tiny workload: k = 12).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SINK_MARGIN = 0.0
N_NEEDLES = 64
N_OUTLIER_CHANNELS = 4


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    n_max: int
    w: int
    pool_kernel: int
    protect: int
    seed: int
    kind: str                      # "gauss_fp32" | "outlier_sink" | "outlier_sink_needle"
    budget_pct: Optional[int] = None   # kept percentage of the non-protected tokens
    evict: Optional[int] = None        # fixed eviction count (tiny workload)
    ragged: Optional[tuple] = None     # (lo, hi) inclusive range of n_b

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def R(self) -> int:
        return self.g * self.w


WORKLOADS = {
    # B=1 Hq=4 Hkv=2 d=16 n=128 w=4, evict 12, pool 3, protect 4; fp32 N(0,1), seeds 42/43/44
    "tiny_d16_n128": WorkloadSpec("tiny_d16_n128", 1, 4, 2, 16, 128, 4, 3, 4, 42,
                                  "gauss_fp32", evict=12),
    # Phi-3-mini-like MHA layer, 10% kept, pool 5
    "phi3mini_mha_d96_n4k": WorkloadSpec("phi3mini_mha_d96_n4k", 1, 32, 32, 96, 4096, 8, 5, 8, 1,
                                         "outlier_sink", budget_pct=10),
    # Llama-3.1-8B-like GQA layer, 10% kept, pool 5, 64 needles
    "llama8b_gqa_d128_n32k": WorkloadSpec("llama8b_gqa_d128_n32k", 1, 32, 8, 128, 32768, 8, 5, 8, 2,
                                          "outlier_sink_needle", budget_pct=10),
    # the same layer at n=128K, 5% kept
    "llama8b_gqa_d128_n128k": WorkloadSpec("llama8b_gqa_d128_n128k", 1, 32, 8, 128, 131072, 8, 5, 8, 3,
                                           "outlier_sink_needle", budget_pct=5),
    # Qwen-like batched layer, ragged n_b ~ U{32768..65536}, 5% kept
    "qwen_gqa7_b4_ragged_n64k": WorkloadSpec("qwen_gqa7_b4_ragged_n64k", 4, 28, 4, 128, 65536, 8, 5, 8, 4,
                                             "outlier_sink_needle", budget_pct=5, ragged=(32768, 65536)),
}

HEADLINE = "llama8b_gqa_d128_n128k"


def evict_count(n_b: int, w: int, budget_pct: int) -> int:
    """k_b = floor((100 - P) * (n_b - w) / 100), integer arithmetic."""
    return ((100 - budget_pct) * (n_b - w)) // 100


def bf16_round(x: np.ndarray) -> torch.Tensor:
    """float32 array -> torch bfloat16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    q: torch.Tensor           # [B, Hq, w, d] bf16 (CPU)
    k: torch.Tensor           # [B, Hkv, n_max, d] bf16 (CPU)
    v: torch.Tensor           # [B, Hkv, n_max, d] bf16 (CPU)
    lengths: torch.Tensor     # [B] int32
    evict_k: torch.Tensor     # [B] int32
    q32: Optional[np.ndarray] = None   # float32 draws (tiny workload only)
    k32: Optional[np.ndarray] = None
    v32: Optional[np.ndarray] = None

    @property
    def shape(self):
        s = self.spec
        return (s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w)

    def kept_len(self) -> np.ndarray:
        return (self.lengths.numpy().astype(np.int64) - self.evict_k.numpy()).astype(np.int32)


def _lse_estimate(n: int, sigma2: np.ndarray) -> np.ndarray:
    """Typical log-sum-exp of n i.i.d. N(0, sigma^2) logits: ln n + sigma^2 / 2
    while sigma <= sqrt(2 ln n), sigma * sqrt(2 ln n) beyond (where the largest
    terms dominate the sum)."""
    ln_n = math.log(n)
    sigma = np.sqrt(sigma2)
    crit = math.sqrt(2.0 * ln_n)
    return np.where(sigma <= crit, ln_n + 0.5 * sigma2, sigma * crit)


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x)


def make_workload(name: str, seed: Optional[int] = None, n_max: Optional[int] = None,
                  keep_fp32: Optional[bool] = None, sink_margin: float = 0.0, v_offset: float = 0.0) -> Workload:
    """Build a named workload.  `seed` overrides the workload's seed; `n_max`
    shrinks the sequence (tests use it for reduced sizes; ragged ranges are
    scaled with it).  `sink_margin` raises the sink's logits by that many nats
    (workloads with a sink); `v_offset` adds a per-head value offset of that
    per-channel spread (module docstring)."""
    spec = WORKLOADS[name]
    if n_max is not None and n_max != spec.n_max:
        rag = spec.ragged
        if rag is not None:
            scale = n_max / spec.n_max
            rag = (max(spec.w + 1, int(rag[0] * scale)), n_max)
        spec = dataclasses.replace(spec, n_max=n_max, ragged=rag)
    if seed is not None:
        spec = dataclasses.replace(spec, seed=seed)
    rng = np.random.default_rng(spec.seed)
    B, Hq, Hkv, d, n, w = spec.B, spec.Hq, spec.Hkv, spec.d, spec.n_max, spec.w
    g = spec.g

    if spec.ragged is not None:
        lengths = rng.integers(spec.ragged[0], spec.ragged[1] + 1, size=B).astype(np.int32)
    else:
        lengths = np.full(B, n, dtype=np.int32)

    q = rng.standard_normal((B, Hq, w, d), dtype=np.float32)
    k = rng.standard_normal((B, Hkv, n, d), dtype=np.float32)
    v = rng.standard_normal((B, Hkv, n, d), dtype=np.float32)

    if spec.kind in ("outlier_sink", "outlier_sink_needle"):
        chan_scale = np.ones((B, Hkv, d), dtype=np.float64)
        for b in range(B):
            for h in range(Hkv):
                ch = rng.choice(d, N_OUTLIER_CHANNELS, replace=False)
                sc = np.exp(rng.uniform(math.log(2.0), math.log(8.0), N_OUTLIER_CHANNELS))
                chan_scale[b, h, ch] = sc
                root = np.sqrt(sc).astype(np.float32)
                k[b, h][:, ch] *= root
                q[b, h * g:(h + 1) * g][..., ch] *= root
        for b in range(B):
            nb = int(lengths[b])
            for h in range(Hkv):
                qg = q[b, h * g:(h + 1) * g].reshape(g * w, d).astype(np.float64)
                sigma2 = ((qg ** 2) * chan_scale[b, h]).sum(axis=1) / d
                target = math.sqrt(d) * (_lse_estimate(nb, sigma2) + SINK_MARGIN + sink_margin)
                # minimum-norm key whose dot product with every window row equals its target
                k0 = qg.T @ np.linalg.solve(qg @ qg.T, target)
                k[b, h, 0] = k0.astype(np.float32)
        if spec.kind == "outlier_sink_needle":
            for b in range(B):
                nb = int(lengths[b])
                for h in range(Hkv):
                    qg = q[b, h * g:(h + 1) * g].reshape(g * w, d).astype(np.float64)
                    pos = rng.choice(np.arange(1, nb - w), N_NEEDLES, replace=False)
                    rows = rng.integers(0, g * w, size=N_NEEDLES)
                    for j, r in zip(pos, rows):
                        u = _unit(qg[r])
                        wv = rng.standard_normal(d)
                        wv -= (wv @ u) * u
                        wv = _unit(wv)
                        nk = float(np.linalg.norm(k[b, h, j].astype(np.float64)))
                        k[b, h, j] = (nk * (0.8 * u + 0.6 * wv)).astype(np.float32)

    if v_offset:
        for b in range(B):
            for h in range(Hkv):
                mu = rng.normal(0.0, v_offset, d)
                ch = rng.choice(d, N_OUTLIER_CHANNELS, replace=False)
                mu[ch] = 4.0 * v_offset * rng.choice([-1.0, 1.0], N_OUTLIER_CHANNELS)
                v[b, h] += mu.astype(np.float32)

    if spec.evict is not None:
        evict = np.full(B, spec.evict, dtype=np.int32)
    else:
        evict = np.array([evict_count(int(nb), w, spec.budget_pct) for nb in lengths], dtype=np.int32)

    keep32 = keep_fp32 if keep_fp32 is not None else (spec.kind == "gauss_fp32")
    wl = Workload(spec=spec, q=bf16_round(q), k=bf16_round(k), v=bf16_round(v),
                  lengths=torch.from_numpy(lengths), evict_k=torch.from_numpy(evict))
    if keep32:
        wl.q32, wl.k32, wl.v32 = q, k, v
    return wl


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 view of its bit patterns (no copy of values)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
