"""GPU parity of the layer-wide selection (AdaDropKV reading: one pool per
sequence over all its KV heads, "DropKV: Decoupling ...", section 5.3 and
Appendix A.3) and of the per-head compaction, against the oracle, through the
C ABI.  Selection is integer work: on the same scores the kept sets must be
identical to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth
from tests._parity import check_kept_layer, check_scores

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _select_layer(scores, lengths, evict_total, protect):
    Bn, H, n = scores.shape
    shape = B.make_shape(Bn, H, H, 8, n, 1)
    ws = torch.empty(B.dropkv_workspace_size(shape), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kept = torch.full((Bn, H, n), -5, dtype=torch.int32, device=DEV)
    kl = torch.full((Bn, H), -1, dtype=torch.int32, device=DEV)
    sc = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).to(DEV)
    for _ in range(2):          # twice: the call clears its own counters
        B.dropkv_select_layer(shape, sc, torch.from_numpy(np.asarray(lengths, np.int32)).to(DEV),
                              torch.from_numpy(np.asarray(evict_total, np.int32)).to(DEV), protect, kept, kl, ws,
                              status)
    code, flags = B.dropkv_read_status(status)
    assert code == 0, "status %d flags 0x%x" % (code, flags)
    return kept.cpu().numpy(), kl.cpu().numpy()


def _check(scores, lengths, evict_total, protect):
    kept, kl = _select_layer(scores, lengths, evict_total, protect)
    rk, rl = oracle.select_layer(scores.astype(np.float64), lengths, evict_total, protect)
    assert np.array_equal(kl, rl), (kl, rl)
    for b in range(scores.shape[0]):
        for h in range(scores.shape[1]):
            assert np.array_equal(kept[b, h, :kl[b, h]], rk[b, h, :kl[b, h]]), "kept set differs (b=%d h=%d)" % (b, h)
            assert np.all(kept[b, h, kl[b, h]:] == -5)


def _protect(s, lengths, protect):
    for b, nb in enumerate(lengths):
        s[b, :, nb - protect:nb] = np.inf
        s[b, :, nb:] = np.nan
    return s


@pytest.mark.parametrize("n", [100, 16384, 40000])
def test_layer_random(n):
    rng = np.random.default_rng(n)
    H = 4
    s = (rng.standard_normal((2, H, n)) ** 2).astype(np.float32)
    lengths = [n, max(9, n // 3)]
    s = _protect(s, lengths, 8)
    _check(s, lengths, [H * (lengths[0] - 8) * 9 // 10, H * (lengths[1] - 8) // 2], 8)


def test_layer_edges():
    rng = np.random.default_rng(1)
    H, n = 3, 30000
    s = (rng.random((4, H, n)) * 1e-6).astype(np.float32)
    lengths = [n, 17, 30001 - 2, n]
    s = _protect(s, lengths, 4)
    _check(s, lengths, [0, H * 13, H * (lengths[2] - 4), 1], 4)


def test_layer_ties_across_heads_and_signed_zero():
    rng = np.random.default_rng(3)
    H, n = 5, 20000
    s = rng.integers(0, 4, size=(2, H, n)).astype(np.float32)
    s[s == 0] = np.where(rng.random(int(np.sum(s == 0))) < 0.5, np.float32(0.0), np.float32(-0.0))
    _check(s, [n, n - 3], [H * 7000, H * 11111], 0)


def test_layer_one_head_equals_per_head_selection():
    """With one KV head the pool is the head: same kept set as dropkv_select."""
    rng = np.random.default_rng(4)
    n = 16387
    s = rng.random((2, 1, n)).astype(np.float32)
    kept, kl = _select_layer(s, [n, 16385], [8000, 16000], 1)
    rk, rl = oracle.select(s.astype(np.float64), [n, 16385], [8000, 16000], 1)
    assert np.array_equal(kl[:, 0], rl)
    for b in range(2):
        assert np.array_equal(kept[b, 0, :kl[b, 0]], rk[b, 0, :rl[b]])


def _layer_path(wl, label):
    s = wl.spec
    et = wl.evict_k.numpy().astype(np.int64) * s.Hkv
    ref = oracle.run_path_layer(wl.q, wl.k, wl.v, wl.lengths, et, s.pool_kernel, s.protect)
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    q, k, v = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    lengths = wl.lengths.to(DEV)
    evt = torch.from_numpy(et.astype(np.int32)).to(DEV)
    op.kept_idx.fill_(-5)
    op.run_layer(q, k, v, lengths, evt)
    op.check()
    lens = wl.lengths.numpy()
    fin = op.scores.cpu().numpy()
    check_scores(fin, ref["final"], lens, label + " final")
    kept, kl = op.kept_idx.cpu().numpy(), op.kept_len_heads.cpu().numpy()
    # integer work on the GPU's own scores: exactly the oracle's selection of them
    own, own_len = oracle.select_layer(np.where(np.isnan(fin), np.inf, fin).astype(np.float64), lens, et, s.protect)
    assert np.array_equal(own_len, kl)
    for b in range(s.B):
        for h in range(s.Hkv):
            assert np.array_equal(own[b, h, :kl[b, h]], kept[b, h, :kl[b, h]])
    band = check_kept_layer(kept, kl, ref["kept_idx"], ref["kept_len"], ref["final"], lens, et)
    # per-head compaction: byte-exact gather of the GPU's own kept rows
    k_out, v_out = op.k_out.cpu(), op.v_out.cpu()
    kc, vc = k.cpu(), v.cpu()
    for b in range(s.B):
        for h in range(s.Hkv):
            idx = torch.from_numpy(kept[b, h, :kl[b, h]].astype(np.int64))
            assert torch.equal(k_out[b, h, :kl[b, h]].view(torch.int16), kc[b, h, idx].view(torch.int16))
            assert torch.equal(v_out[b, h, :kl[b, h]].view(torch.int16), vc[b, h, idx].view(torch.int16))
    print("%s: %d band slots; kept per head %s" % (label, band, kl.tolist()))


@pytest.mark.parametrize("name,n_max", [("tiny_d16_n128", None), ("phi3mini_mha_d96_n4k", 1000),
                                        ("qwen_gqa7_b4_ragged_n64k", 3000)])
def test_layer_path_reduced(name, n_max):
    wl = synth.make_workload(name, n_max=n_max) if n_max else synth.make_workload(name)
    _layer_path(wl, "layer %s" % name)


@pytest.mark.parametrize("name", ["llama8b_gqa_d128_n128k", "qwen_gqa7_b4_ragged_n64k"])
def test_layer_path_full_size(name):
    _layer_path(synth.make_workload(name), "layer " + name)
