"""GPU parity where the method is numerically delicate.

A dominant key (an attention sink) that carries nearly all of a row's mass
makes 1 - p_j and |a - v_j| tiny differences of large quantities: the
pages' closed form p/(1-p) (a - v_j) ("DropKV: Exact single-entry
output-perturbation scoring", Core equation) has to be evaluated without
that cancellation, and an input whose p_j rounds to 1 has to be rejected,
not patched (same page, Algorithm 1 summary).  Values that share a large
common offset make |v|^2 far larger than |a - v|^2, the other place where an
expanded distance loses digits.  Every case is compared element by element
with the fp64 oracle at the usual bound (relative 2e-3, absolute 1e-6, and
the scale-aware bound), and the kept sets and compaction as everywhere else.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth
from tests._gpu import DEV, _compare, _custom, _run, _run_custom
from tests._parity import deletion_score

pytestmark = pytest.mark.gpu

SINK_LEVELS = [0.9, 0.99, 0.999, 0.9999, 1 - 1e-6]


def _margin(p0):
    """Logit margin (nats) that puts about p0 of a row's mass on the sink."""
    return math.log(p0 / (1.0 - p0))


def _sink_mass(wl, ref, pos=0):
    """Per-row probability of key `pos` from the oracle's statistics."""
    s = wl.spec
    q, k = wl.q.double().numpy(), wl.k.double().numpy()
    out = []
    for b in range(s.B):
        for hq in range(s.Hq):
            x = q[b, hq] @ k[b, hq // s.g, pos] / math.sqrt(s.d)
            out.append(np.exp(x - ref["m"][b, hq]) / ref["l"][b, hq])
    return np.concatenate(out)


def _check_sink(name, p0, n_max=None, v_offset=0.0):
    wl = synth.make_workload(name, n_max=n_max, sink_margin=_margin(p0), v_offset=v_offset)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    pm = _sink_mass(wl, ref)
    # the workload really is in the regime: most rows put about p0 on the sink
    assert np.median(pm) >= 1 - 20 * (1 - p0), np.median(pm)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "%s sink p0=%g (median %.7f, max %.9f)" % (name, p0, np.median(pm), pm.max()))


@pytest.mark.parametrize("p0", SINK_LEVELS)
def test_sink_mass_llama8b_n32k(p0):
    _check_sink("llama8b_gqa_d128_n32k", p0)


@pytest.mark.parametrize("p0", SINK_LEVELS)
def test_sink_mass_llama8b_n128k(p0):
    _check_sink("llama8b_gqa_d128_n128k", p0)


@pytest.mark.parametrize("p0", [0.999, 1 - 1e-6])
def test_sink_mass_ragged_gqa7(p0):
    """Ragged batch: the dominant splits follow pass 1's length-proportional share."""
    _check_sink("qwen_gqa7_b4_ragged_n64k", p0, n_max=20000)


@pytest.mark.parametrize("p0", [0.99, 1 - 1e-6])
def test_sink_mass_mha_d96(p0):
    _check_sink("phi3mini_mha_d96_n4k", p0)


def _tiny_with_sink(p0, seed):
    """The tiny workload's shape with key 0 set so that every window row puts
    about p0 of its mass on it (minimum-norm key with the required logits)."""
    wl = synth.make_workload("tiny_d16_n128", seed=seed)
    s = wl.spec
    q = wl.q.double().numpy()
    k = wl.k.double().numpy()
    for h in range(s.Hkv):
        qg = q[0, h * s.g:(h + 1) * s.g].reshape(s.R, s.d)
        rest = np.empty(s.R)
        for r in range(s.R):
            pos = s.n_max - s.w + r % s.w
            x = k[0, h, 1:pos + 1] @ qg[r] / math.sqrt(s.d)
            rest[r] = np.log(np.sum(np.exp(x - x.max()))) + x.max()
        target = math.sqrt(s.d) * (rest + _margin(p0))
        k[0, h, 0] = qg.T @ np.linalg.solve(qg @ qg.T, target)
    return synth.Workload(spec=s, q=wl.q, k=synth.bf16_round(k.astype(np.float32)), v=wl.v,
                          lengths=wl.lengths, evict_k=wl.evict_k)


@pytest.mark.parametrize("p0", SINK_LEVELS)
@pytest.mark.parametrize("seed", [42, 43])
def test_sink_mass_tiny(p0, seed):
    wl = _tiny_with_sink(p0, seed)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    pm = _sink_mass(wl, ref)
    assert np.median(pm) >= 1 - 20 * (1 - p0)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "tiny sink p0=%g seed %d" % (p0, seed))


def test_sink_beyond_double_precision_is_singular():
    """Sink logits about 40 nats above the rest: 1 - p is near 4e-18, so p
    rounds to 1 in double precision.  The oracle rejects the input and the GPU
    reports SINGULAR (and +inf for the key), rather than a patched score."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=6000, sink_margin=40.0)
    s = wl.spec
    with pytest.raises(oracle.SingularInput):
        oracle.score(wl.q, wl.k, wl.v, wl.lengths.numpy(), s.pool_kernel, s.protect)
    op, _, _, _ = _run_nocheck(wl)
    code, flags = B.dropkv_read_status(op.status)
    assert code == 3 and flags & B.FLAG_SINGULAR
    assert torch.isinf(op.raw_scores[0, :, 0]).all()


def test_sink_at_one_minus_1e9():
    """Sink logits about 20.7 nats above the rest (1 - p near 1e-9): the
    oracle's fp64 closed form is still exact to about 1e-7 here (its sum of the
    other keys' mass keeps enough digits), and the GPU matches it."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=6000, sink_margin=20.7)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "sink 20.7 nats")


def test_sink_just_short_of_double_precision():
    """About 30 nats (1 - p near 1e-13): p does not round to 1 in double
    precision, so the input is scored.  The closed form would keep three
    digits here; the oracle takes the sink in the deletion form and so does
    the GPU's dominant-key path.  Every output against the oracle, and the
    sink's score also against fp64 deletion from the logits."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=6000, sink_margin=30.0)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, flags = _run(wl)
    _compare(wl, op, k, v, ref, "sink 30 nats")
    raw = op.raw_scores.cpu().numpy()
    dl = deletion_score(*(t.double().numpy() for t in (wl.q, wl.k, wl.v)), wl.lengths.numpy(), j=0)
    np.testing.assert_allclose(raw[:, :, 0], dl, rtol=2e-3)


def _run_nocheck(wl):
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    q, k, v = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    op.run(q, k, v, wl.lengths.to(DEV), wl.evict_k.to(DEV))
    return op, k, v, None


def test_dominant_keys_in_different_splits():
    """Each query head of a group leans on its own key, placed in a different
    pass-1 split (one near the start, two mid-range, one in the last tile
    before the window): several CTAs of the unit handle dominant rows, next to
    rows with no dominant key."""
    n, d = 128 * 152 + 77, 64
    q, k, v, lens = _custom(1, 5, 1, d, n, 2, seed=51)
    positions = [3, 128 * 40 + 9, 128 * 97 + 100, n - 2 - 64]
    target = 17.0 + math.log(n) + 0.5       # about 17 nats above the log-sum-exp of the other keys
    for hl, pos in enumerate(positions):
        qs = q[0, hl].sum(axis=0)               # both window rows of query head hl
        # q_t . k / sqrt(d) close to `target` for t = 0, 1 (q_t . qs is about qs . qs / 2)
        k[0, 0, pos] = target * math.sqrt(d) * 2.0 / float(qs @ qs) * qs
    _run_custom(q, k, v, lens, [n // 2], 5, 2)


def test_mixed_dominated_and_plain_heads_ragged():
    """A ragged batch where half of the KV heads have a sink at p near 0.9999
    and the others none: dynamic and static/dominant CTAs in one launch."""
    wl = synth.make_workload("qwen_gqa7_b4_ragged_n64k", n_max=9000, sink_margin=_margin(0.9999))
    k = wl.k.clone()
    k[:, 2:, 0] = k[:, 2:, 1]                      # heads 2, 3: no sink
    wl = synth.Workload(spec=wl.spec, q=wl.q, k=k, v=wl.v, lengths=wl.lengths, evict_k=wl.evict_k)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, kd, vd, _ = _run(wl)
    _compare(wl, op, kd, vd, ref, "mixed heads")


def test_one_call_equals_three_calls_with_a_sink():
    """The dominant path is deterministic: dropkv_evict and the three separate
    calls write the same bytes."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", sink_margin=_margin(0.9999))
    s = wl.spec
    q, k, v = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    lengths, ev = wl.lengths.to(DEV), wl.evict_k.to(DEV)
    outs = []
    for fused in (True, False, True):
        op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
        for t in (op.scores, op.raw_scores):      # entries the calls leave untouched are compared too
            t.fill_(-7.25)
        op.kept_idx.fill_(-5)
        op.k_out.zero_()
        op.v_out.zero_()
        (op.run if fused else op.run_separate)(q, k, v, lengths, ev)
        op.check()
        outs.append([t.clone() for t in (op.scores, op.raw_scores, op.kept_idx, op.kept_len, op.k_out, op.v_out)])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.int8), b.view(torch.int8))


# ------------------------------------------------------------ value offsets
@pytest.mark.parametrize("sigma", [4.0, 16.0])
def test_value_offset_llama8b_n32k(sigma):
    wl = synth.make_workload("llama8b_gqa_d128_n32k", v_offset=sigma)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "value offset %g" % sigma)


def test_value_offset_llama8b_n128k():
    wl = synth.make_workload("llama8b_gqa_d128_n128k", v_offset=8.0)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "value offset 8, n=128K")


def test_value_offset_with_sink():
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=12000, sink_margin=_margin(0.9999), v_offset=8.0)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "value offset 8 with a sink")
