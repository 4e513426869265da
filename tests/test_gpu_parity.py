"""GPU parity of the CUDA path against the oracle, through the C ABI.

Inputs are the seeded workloads; the oracle sees exactly the bf16 values the
GPU reads.  Every workload runs at its full size, plus reduced sizes that
still span several tiles with a ragged tail and the edge cases of the method.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth
from tests._gpu import DEV, SENTINEL, _compare, _custom, _run, _run_custom
from tests._parity import check_scores

pytestmark = pytest.mark.gpu

@pytest.mark.parametrize("seed", [42, 43, 44])
def test_tiny_workload(seed):
    wl = synth.make_workload("tiny_d16_n128", seed=seed)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "tiny seed %d" % seed)


@pytest.mark.parametrize("name,n_max", [
    ("phi3mini_mha_d96_n4k", 1000),
    ("llama8b_gqa_d128_n32k", 2 * 128 * 19 + 57),
    ("qwen_gqa7_b4_ragged_n64k", 3000),
])
def test_reduced_sizes_ragged_tail(name, n_max):
    wl = synth.make_workload(name, n_max=n_max)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, "%s n=%d" % (name, n_max))


@pytest.mark.parametrize("name", [
    "phi3mini_mha_d96_n4k",
    "llama8b_gqa_d128_n32k",
    "llama8b_gqa_d128_n128k",
    "qwen_gqa7_b4_ragged_n64k",
])
def test_full_size_workloads(name):
    wl = synth.make_workload(name)
    s = wl.spec
    ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(wl)
    _compare(wl, op, k, v, ref, name)


@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, d, n, w, pool, protect, evict)
    (1, 1, 1, 64, 128, 1, 1, 0, [0]),          # w=1, g=1, pool 1, nothing evicted
    (1, 2, 1, 32, 77, 3, 1, 0, [74]),          # n < one tile, evict every unprotected slot
    (1, 8, 2, 128, 300, 4, 7, 4, [150]),       # g=4, several tiles, ragged tail
    (2, 4, 4, 96, 513, 2, 3, 2, [400, 1]),     # MHA, d=96
    (1, 16, 1, 128, 1025, 4, 5, 4, [1000]),    # R=64 (largest supported group x window)
    (1, 3, 1, 8, 260, 5, 9, 5, [100]),         # d=8, R=15
])
def test_edge_shapes(case):
    B, Hq, Hkv, d, n, w, pool, protect, evict = case
    q, k, v, lens = _custom(B, Hq, Hkv, d, n, w, seed=sum(case[:6]))
    _run_custom(q, k, v, lens, evict, pool, protect)


def test_ragged_lengths_with_nan_padding():
    q, k, v, lens = _custom(3, 4, 2, 64, 700, 4, seed=5, lengths=[700, 129, 333])
    _run_custom(q, k, v, lens, [600, 100, 0], 5, 4)


def test_logit_jump_inside_a_chunk():
    """Two keys about 20 nats above every other logit, each in the third tile of
    a different CTA's range: the CTA's running exponent reference has to move
    mid-range and its accumulator be rescaled.  Each big key ends near p = 0.5."""
    n = 128 * 152 * 4
    q, k, v, lens = _custom(1, 1, 1, 64, n, 2, seed=9)
    q[0, 0, 1] = q[0, 0, 0]
    qn = q[0, 0, 0] / np.linalg.norm(q[0, 0, 0])
    big = 20.0 * np.sqrt(64) / np.linalg.norm(q[0, 0, 0])
    for pos in (128 * (4 * 10 + 2) + 5, 128 * (4 * 50 + 3) + 77):
        k[0, 0, pos] = big * qn
    _run_custom(q, k, v, lens, [n // 2], 3, 2)


def test_ties_and_protection():
    """Identical keys and values give equal scores: ties must be evicted lowest position first."""
    q, k, v, lens = _custom(1, 2, 1, 32, 640, 2, seed=4)
    k[0, 0, 100:400] = k[0, 0, 100]
    v[0, 0, 100:400] = v[0, 0, 100]
    _run_custom(q, k, v, lens, [250], 1, 2)


@pytest.mark.parametrize("name,n_max,pool", [("tiny_d16_n128", None, None), ("phi3mini_mha_d96_n4k", None, None),
                                              ("qwen_gqa7_b4_ragged_n64k", None, None),
                                              ("llama8b_gqa_d128_n32k", 40000, 63),
                                              ("llama8b_gqa_d128_n32k", 140000, None)])
def test_one_call_equals_three_calls(name, n_max, pool):
    """dropkv_evict (pooling inside the cluster selection for heads of at most
    8 chunks; pool kernel + multi-kernel selection beyond) writes exactly what
    dropkv_score, dropkv_select and dropkv_compact write in sequence."""
    wl = synth.make_workload(name, n_max=n_max) if n_max else synth.make_workload(name)
    s = wl.spec
    kappa = pool or s.pool_kernel
    q, k, v = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    lengths, ev = wl.lengths.to(DEV), wl.evict_k.to(DEV)
    outs = []
    for fused in (True, False):
        op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, kappa, s.protect, device=DEV)
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


def _sweep_cases(count, seed):
    """Seeded random shapes over the supported range: g, w with R = g w <= 64,
    d a multiple of 8 up to 128, ragged lengths, any odd pooling kernel."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < count:
        Hkv = int(rng.integers(1, 4))
        g = int(rng.integers(1, 9))
        w = int(rng.integers(1, 9))
        if g * w > 64:
            continue
        d = int(rng.choice([8, 16, 24, 64, 96, 120, 128]))
        B = int(rng.integers(1, 4))
        n = int(rng.integers(w + 1, 3000))
        lens = rng.integers(max(w, 1), n + 1, size=B)
        protect = int(rng.integers(0, w + 1))
        pool = int(rng.choice([1, 3, 5, 7, 9, 63]))
        evict = [int(rng.integers(0, max(1, int(L) - protect) + 1)) for L in lens]
        cases.append((B, g * Hkv, Hkv, d, n, w, pool, protect, lens.tolist(), evict))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(12, 2026))
def test_random_shape_sweep(case):
    B, Hq, Hkv, d, n, w, pool, protect, lens, evict = case
    q, k, v, lengths = _custom(B, Hq, Hkv, d, n, w, seed=sum(lens) + d, lengths=lens)
    _run_custom(q, k, v, lengths, evict, pool, protect)


def test_short_sequences():
    """Sequences of w + 1 and w + 2 tokens (the first window row sees two
    keys, everything or all but one slot protected) next to a normal one."""
    q, k, v, lens = _custom(3, 4, 2, 64, 300, 6, seed=17, lengths=[7, 300, 8])
    _run_custom(q, k, v, lens, [1, 200, 0], 3, 6)


def test_sequence_of_w_tokens_is_singular():
    """With n_b = w the first window row sees a single key, so p = 1 and exact
    removal is singular: the oracle rejects the input and the GPU reports
    SINGULAR (the method's degenerate case, not patched)."""
    q, k, v, lens = _custom(2, 4, 2, 64, 300, 6, seed=19, lengths=[6, 300])
    with pytest.raises(oracle.SingularInput):
        oracle.score(synth.bf16_round(q), synth.bf16_round(k), synth.bf16_round(v), lens, 3, 6)
    op = DropKV(2, 4, 2, 64, 300, 6, 3, 6, device=DEV)
    op.run(synth.bf16_round(q).to(DEV), synth.bf16_round(k).to(DEV), synth.bf16_round(v).to(DEV),
           torch.from_numpy(lens).to(DEV), torch.tensor([0, 100], dtype=torch.int32, device=DEV))
    code, flags = B.dropkv_read_status(op.status)
    assert code == 3 and flags & B.FLAG_SINGULAR


def test_one_million_tokens():
    """n = 2^20 in one KV head (64 selection chunks: the multi-kernel radix
    path; 8192 pass-1 tiles over every SM)."""
    n = 1 << 20
    q, k, v, lens = _custom(1, 1, 1, 128, n, 8, seed=23)
    _run_custom(q, k, v, lens, [n * 9 // 10], 5, 8)


# The passes share their one-wave grid out over the KV heads in proportion to
# the sequence lengths (read on the device).  These batches put that mapping
# far from the even split: one long sequence beside short ones, more than 32
# sequences (several warp-wide chunks of the prefix scan), and more KV heads
# than SMs (one CTA each).
@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, d, n, w, lengths or None for random, seed)
    (5, 4, 2, 64, 20000, 4, [20000, 300, 129, 5000, 9], 31),
    (37, 8, 4, 32, 700, 3, None, 32),
    (40, 4, 4, 16, 400, 2, None, 33),
])
def test_grid_share_across_ragged_heads(case):
    B, Hq, Hkv, d, n, w, lens, seed = case
    if lens is None:
        lens = np.random.default_rng(seed).integers(w + 1, n + 1, size=B).tolist()
    q, k, v, lengths = _custom(B, Hq, Hkv, d, n, w, seed=seed, lengths=lens)
    evict = [int(L) // 2 for L in lens]
    _run_custom(q, k, v, lengths, evict, 3, w)


def test_invalid_lengths_beside_valid_ones():
    """Lengths below w or above n_max are flagged and their heads skipped; the
    valid sequence between them is scored as if it were alone."""
    Bn, Hq, Hkv, d, n, w = 3, 4, 2, 64, 3000, 4
    q, k, v, _ = _custom(Bn, Hq, Hkv, d, n, w, seed=35)
    qb, kb, vb = synth.bf16_round(q), synth.bf16_round(k), synth.bf16_round(v)
    op = DropKV(Bn, Hq, Hkv, d, n, w, 3, w, device=DEV)
    op.scores.fill_(SENTINEL)
    lens = torch.tensor([3, 2500, 1 << 30], dtype=torch.int32, device=DEV)
    op.score(qb.to(DEV), kb.to(DEV), vb.to(DEV), lens)
    code, flags = B.dropkv_read_status(op.status)
    assert code == 7 and flags & B.FLAG_BAD_LENGTH
    ref = oracle.score(qb[1:2], kb[1:2], vb[1:2], np.array([2500], dtype=np.int32), 3, w)
    check_scores(op.scores[1:2].cpu().numpy(), ref["final"], [2500])


def test_single_sequence_far_shorter_than_the_cache():
    """One sequence of 300 tokens in a 40000-slot cache: the one-sequence grid
    gives the head floor(SMs / Hkv) CTAs from the capacity, most of which find
    no tile of the sequence and publish an empty split state."""
    q, k, v, lens = _custom(1, 8, 2, 64, 40000, 4, seed=41, lengths=[300])
    _run_custom(q, k, v, lens, [150], 5, 4)
