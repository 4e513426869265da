"""Decode-time re-scoring input: the cache one prefill eviction leaves, grown
by m decode tokens.

The pages leave a decode-time kernel as future work (DropKV paper, section 6,
"Limitations and future work").  The reading built here: the prefill step
(score -> select -> compact) keeps n_b - k_b rows per KV head, in position
order; decoding appends m new keys and values to that compacted cache; the
observation window moves to the newest w positions, that is the last w - m
queries of the previous window followed by the m new ones when m < w, else the
last w of the new ones; the grown cache is then scored with the same kernels
and m rows are evicted again, so the cache stays at its budget.  The new
tokens' Q/K/V are seeded N(0, 1) bf16 draws; no data comes from a model.

grow_after_eviction() runs the prefill step on the GPU through the library and
returns the grown cache as a host workload, ready for the same calls.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import synth
from .api import DropKV


def grow_after_eviction(wl: synth.Workload, m: int, seed: int, device) -> synth.Workload:
    """Prefill eviction of `wl` on `device`, then m decode tokens appended and
    the window moved.  The returned workload holds host tensors: q [B,Hq,w,d],
    k/v [B,Hkv,max_b(kept_b) + m,d] (rows past kept_b + m are zero), lengths
    kept_b + m and evict_k = m."""
    if m < 1:
        raise ValueError("m must be at least 1")
    s = wl.spec
    kept = wl.kept_len()
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, out_rows=int(kept.max()),
                device=device, kind="dropkv")
    op.run(wl.q.to(device), wl.k.to(device), wl.v.to(device), wl.lengths.to(device), wl.evict_k.to(device))
    op.check()
    got = op.kept_len.cpu().numpy()
    if not np.array_equal(got, kept):
        raise RuntimeError("prefill eviction kept %s rows, expected %s" % (got.tolist(), kept.tolist()))
    return append_decode_tokens(wl, op.k_out.cpu(), op.v_out.cpu(), m, seed)


def append_decode_tokens(wl: synth.Workload, k_kept: torch.Tensor, v_kept: torch.Tensor, m: int,
                         seed: int) -> synth.Workload:
    """The grown cache from a compacted one: k_kept/v_kept [B,Hkv,>=kept_b,d]
    host tensors holding each head's kept rows in position order (kept_b =
    n_b - k_b of `wl`), then m seeded decode tokens per sequence."""
    s = wl.spec
    kept = wl.kept_len()
    rng = np.random.default_rng(seed)
    k_new = synth.bf16_round(rng.standard_normal((s.B, s.Hkv, m, s.d)).astype(np.float32))
    v_new = synth.bf16_round(rng.standard_normal((s.B, s.Hkv, m, s.d)).astype(np.float32))
    q_new = synth.bf16_round(rng.standard_normal((s.B, s.Hq, m, s.d)).astype(np.float32))
    n = int(kept.max()) + m
    k = torch.zeros(s.B, s.Hkv, n, s.d, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for b in range(s.B):
        kb = int(kept[b])
        k[b, :, :kb] = k_kept[b, :, :kb]
        v[b, :, :kb] = v_kept[b, :, :kb]
        k[b, :, kb:kb + m] = k_new[b]
        v[b, :, kb:kb + m] = v_new[b]
    if m >= s.w:
        q = q_new[:, :, m - s.w:]
    else:
        q = torch.cat([wl.q[:, :, m:], q_new], dim=2)
    lengths = torch.from_numpy((kept + m).astype(np.int32))
    base = s.name.split(":decode")[0]
    spec = dataclasses.replace(s, name="%s:decode%d" % (base, m), n_max=n, seed=seed, evict=m, budget_pct=None,
                               ragged=None)
    return synth.Workload(spec=spec, q=q.contiguous(), k=k, v=v, lengths=lengths,
                          evict_k=torch.full((s.B,), m, dtype=torch.int32))
