"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on a
seeded workload and compare every output with the oracle (scores, window
statistics, kept sets, compaction)."""
import numpy as np
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, synth
from tests._parity import check_kept, check_scores

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
SENTINEL = -7.25


def _run(wl, poison=True, out_rows=None, kind="dropkv"):
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, out_rows=out_rows, device=DEV,
                kind=kind)
    k, v = wl.k.clone(), wl.v.clone()
    if poison:
        for b in range(s.B):
            nb = int(wl.lengths[b])
            k[b, :, nb:] = float("nan")
            v[b, :, nb:] = float("nan")
    q, k, v = wl.q.to(DEV), k.to(DEV), v.to(DEV)
    lengths, ev = wl.lengths.to(DEV), wl.evict_k.to(DEV)
    op.scores.fill_(SENTINEL)
    op.raw_scores.fill_(SENTINEL)
    op.kept_idx.fill_(-5)
    op.run(q, k, v, lengths, ev)
    flags = op.check()
    return op, k, v, flags


def _compare(wl, op, kdev, vdev, ref, label, kind="dropkv"):
    s = wl.spec
    lengths = wl.lengths.numpy()
    raw = op.raw_scores.cpu().numpy()
    fin = op.scores.cpu().numpy()
    w_raw = check_scores(raw, ref["raw"], lengths, label + " raw")
    w_fin = check_scores(fin, ref["final"], lengths, label + " final")
    for b in range(s.B):          # slots past n_b are never written
        nb = int(lengths[b])
        assert np.all(fin[b, :, nb:] == SENTINEL) and np.all(raw[b, :, nb:] == SENTINEL)
    lse, a = (t.cpu().numpy() for t in op.window_stats())
    ref_lse = (ref["m"] + np.log(ref["l"])).reshape(lse.shape)
    ref_a = ref["a"].reshape(a.shape)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-5, atol=1e-4)
    if kind == "dropkv":        # the SnapKV path does not compute a
        scale_a = np.abs(ref_a).max(axis=-1, keepdims=True)
        assert np.all(np.abs(a - ref_a) <= 1e-4 * scale_a + 1e-6), float(np.max(np.abs(a - ref_a) / scale_a))
    kept = op.kept_idx.cpu().numpy()
    kl = op.kept_len.cpu().numpy()
    # selection is integer work: on the GPU's own scores it must equal a stable sort exactly
    own_kept, own_len = oracle.select(np.where(np.isnan(fin), np.inf, fin).astype(np.float64), lengths,
                                      wl.evict_k.numpy(), s.protect)
    assert np.array_equal(own_len, kl)
    for b in range(s.B):
        assert np.array_equal(own_kept[b, :, :kl[b]], kept[b, :, :kl[b]]), "select != stable sort of GPU scores"
    band = check_kept(kept, kl, ref["kept_idx"], ref["kept_len"], ref["final"], lengths, wl.evict_k.numpy())
    # compaction: byte-exact gather of the GPU's own kept rows
    k_out, v_out = op.k_out.cpu(), op.v_out.cpu()
    kc, vc = kdev.cpu(), vdev.cpu()
    for b in range(s.B):
        for h in range(s.Hkv):
            idx = torch.from_numpy(kept[b, h, :kl[b]].astype(np.int64))
            assert torch.equal(k_out[b, h, :kl[b]].view(torch.int16), kc[b, h, idx].view(torch.int16))
            assert torch.equal(v_out[b, h, :kl[b]].view(torch.int16), vc[b, h, idx].view(torch.int16))
            assert np.all(kept[b, h, kl[b]:] == -5)
    print("%s: worst raw %.3f / final %.3f of tolerance, %d band tokens" % (label, w_raw, w_fin, band))


def _custom(B, Hq, Hkv, d, n, w, seed=0, lengths=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, w, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, n, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, n, d)).astype(np.float32)
    lens = np.full(B, n, dtype=np.int32) if lengths is None else np.asarray(lengths, dtype=np.int32)
    return q, k, v, lens


def _run_custom(q, k, v, lens, evict, pool, protect):
    wl = synth.Workload(spec=synth.WorkloadSpec("custom", q.shape[0], q.shape[1], k.shape[1], q.shape[3],
                                                k.shape[2], q.shape[2], pool, protect, 0, "custom"),
                        q=synth.bf16_round(q), k=synth.bf16_round(k), v=synth.bf16_round(v),
                        lengths=torch.from_numpy(lens), evict_k=torch.from_numpy(np.asarray(evict, dtype=np.int32)))
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, pool, protect)
    op, kd, vd, flags = _run(wl)
    _compare(wl, op, kd, vd, ref, "custom")
    return op, flags


