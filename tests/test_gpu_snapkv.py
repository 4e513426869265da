"""GPU parity of the SnapKV score kind (the attention-only baseline of
"DropKV: Decoupling Residual-Output Perturbation for Near-Optimal KV-Cache
Eviction", Appendix B, Table 14) against the oracle, through the C ABI.

Same inputs, windows, pooling, protection, selection and compaction as the
DropKV path; the score of key j is the window sum of its attention
probabilities, averaged over the query heads of the group.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, synth
from tests.test_gpu_parity import DEV, SENTINEL, _compare, _custom, _run

pytestmark = pytest.mark.gpu


def _check(wl, label):
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect, kind="snapkv")
    op, k, v, _ = _run(wl, kind="snapkv")
    _compare(wl, op, k, v, ref, label, kind="snapkv")
    # the raw scores of a KV head sum to w (every window row's probabilities sum to 1)
    raw = op.raw_scores.cpu().numpy().astype(np.float64)
    for b in range(s.B):
        nb = int(wl.lengths[b])
        np.testing.assert_allclose(raw[b, :, :nb].sum(axis=-1), s.w, rtol=2e-3)


@pytest.mark.parametrize("seed", [42, 43, 44])
def test_snapkv_tiny(seed):
    _check(synth.make_workload("tiny_d16_n128", seed=seed), "snapkv tiny %d" % seed)


@pytest.mark.parametrize("name,n_max", [
    ("phi3mini_mha_d96_n4k", 1000),
    ("llama8b_gqa_d128_n32k", 2 * 128 * 19 + 57),
    ("qwen_gqa7_b4_ragged_n64k", 3000),
])
def test_snapkv_reduced_sizes(name, n_max):
    _check(synth.make_workload(name, n_max=n_max), "snapkv %s n=%d" % (name, n_max))


@pytest.mark.parametrize("name", [
    "phi3mini_mha_d96_n4k",
    "llama8b_gqa_d128_n32k",
    "llama8b_gqa_d128_n128k",
    "qwen_gqa7_b4_ragged_n64k",
])
def test_snapkv_full_size(name):
    _check(synth.make_workload(name), "snapkv " + name)


@pytest.mark.parametrize("case", [
    (1, 2, 1, 32, 77, 3, 1, 0, [74]),
    (2, 4, 4, 96, 513, 2, 3, 2, [400, 1]),
    (1, 16, 1, 128, 1025, 4, 5, 4, [1000]),
    (1, 3, 1, 8, 260, 5, 9, 5, [100]),
])
def test_snapkv_edge_shapes(case):
    B, Hq, Hkv, d, n, w, pool, protect, evict = case
    q, k, v, lens = _custom(B, Hq, Hkv, d, n, w, seed=sum(case[:6]))
    wl = synth.Workload(spec=synth.WorkloadSpec("custom", B, Hq, Hkv, d, n, w, pool, protect, 0, "custom"),
                        q=synth.bf16_round(q), k=synth.bf16_round(k), v=synth.bf16_round(v),
                        lengths=torch.from_numpy(lens), evict_k=torch.from_numpy(np.asarray(evict, dtype=np.int32)))
    _check(wl, "snapkv custom")


def test_snapkv_accepts_the_singular_input():
    """One key dominates every window row (p_j rounds to 1): DropKV reports
    SINGULAR, SnapKV scores it w and everything else 0."""
    q, k, v, lens = _custom(1, 1, 1, 16, 256, 2, seed=9)
    q[..., 0] = 100.0
    k[0, 0, 5, 0] = 100.0
    k[0, 0, np.arange(256) != 5, 0] = 0.0
    qd, kd, vd = (synth.bf16_round(x).to(DEV) for x in (q, k, v))
    lengths = torch.from_numpy(lens).to(DEV)
    ev = torch.tensor([100], dtype=torch.int32, device=DEV)
    op = DropKV(1, 1, 1, 16, 256, 2, 1, 0, device=DEV, kind="snapkv")
    op.run(qd, kd, vd, lengths, ev)
    op.check()
    raw = op.raw_scores.cpu().numpy()[0, 0]
    assert raw[5] == pytest.approx(2.0, rel=1e-5)
    assert np.all(raw[np.arange(256) != 5] == 0.0)


@pytest.mark.parametrize("name,n_max", [("qwen_gqa7_b4_ragged_n64k", None), ("llama8b_gqa_d128_n32k", 140000)])
def test_snapkv_one_call_equals_three_calls(name, n_max):
    wl = synth.make_workload(name, n_max=n_max) if n_max else synth.make_workload(name)
    s = wl.spec
    q, k, v = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    lengths, ev = wl.lengths.to(DEV), wl.evict_k.to(DEV)
    outs = []
    for fused in (True, False):
        op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV, kind="snapkv")
        for t in (op.scores, op.raw_scores):
            t.fill_(SENTINEL)
        op.kept_idx.fill_(-5)
        op.k_out.zero_()
        op.v_out.zero_()
        (op.run if fused else op.run_separate)(q, k, v, lengths, ev)
        op.check()
        outs.append([t.clone() for t in (op.scores, op.raw_scores, op.kept_idx, op.kept_len, op.k_out, op.v_out)])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int8), b.view(torch.int8))
