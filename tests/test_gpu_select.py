"""Bit-exact parity of dropkv_select with the oracle's stable sort, on crafted
score arrays that drive every branch of both selection paths: heads of up to
eight 16384-slot chunks are selected inside one thread-block cluster (digit
histograms merged across the cluster, ties ranked by position across its
CTAs); longer heads take the multi-kernel radix path (few ties, a 24-bit
prefix shared by a few slots, large tie sets, a level-1 bin larger than the
candidate buffer).  Also signed zeros, ragged lengths and the k = 0 /
k = n - protect edges.  Selection is integer work, so the kept sets must be
identical."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import _binding as B

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _select(scores, lengths, evict, protect):
    Bn, H, n = scores.shape
    shape = B.make_shape(Bn, H, H, 8, n, 1)
    ws = torch.empty(B.dropkv_workspace_size(shape), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kept = torch.full((Bn, H, n), -5, dtype=torch.int32, device=DEV)
    kl = torch.zeros(Bn, dtype=torch.int32, device=DEV)
    sc = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).to(DEV)
    B.dropkv_select(shape, sc, torch.from_numpy(np.asarray(lengths, np.int32)).to(DEV),
                    torch.from_numpy(np.asarray(evict, np.int32)).to(DEV), protect, kept, kl, ws, status)
    code, flags = B.dropkv_read_status(status)
    assert code == 0, "status %d flags 0x%x" % (code, flags)
    return kept.cpu().numpy(), kl.cpu().numpy()


def _check(scores, lengths, evict, protect):
    kept, kl = _select(scores, lengths, evict, protect)
    rk, rl = oracle.select(scores.astype(np.float64), lengths, evict, protect)
    assert np.array_equal(kl, rl)
    for b in range(scores.shape[0]):
        assert np.array_equal(kept[b, :, :kl[b]], rk[b, :, :kl[b]]), "kept set differs (b=%d)" % b
        assert np.all(kept[b, :, kl[b]:] == -5)


def _protect(scores, lengths, protect):
    for b, nb in enumerate(lengths):
        scores[b, :, nb - protect:nb] = np.inf
        scores[b, :, nb:] = np.nan
    return scores


@pytest.mark.parametrize("n", [100, 16383, 16384, 50001])
def test_random_scores(n):
    rng = np.random.default_rng(n)
    s = (rng.standard_normal((2, 3, n)) ** 2).astype(np.float32)
    lengths = [n, max(9, n // 3)]
    s = _protect(s, lengths, 8)
    _check(s, lengths, [(lengths[0] - 8) * 9 // 10, (lengths[1] - 8) // 2], 8)


def test_k_edges_and_ragged():
    rng = np.random.default_rng(1)
    n = 40000
    s = (rng.random((3, 2, n)) * 1e-6).astype(np.float32)
    lengths = [n, 17, 30001]
    s = _protect(s, lengths, 4)
    _check(s, lengths, [0, 13, 29997], 4)


def test_few_slots_share_the_k_th_prefix():
    rng = np.random.default_rng(2)
    n = 30000
    base = (rng.random(n) + 1.0).astype(np.float32)
    # values that differ only in the last mantissa bits around the cut
    s = np.tile(base, (1, 2, 1))
    s[0, 0, 100:140] = np.float32(1.5) + np.arange(40, dtype=np.float32) * np.float32(2 ** -23)
    _check(s, [n], [n // 2], 0)


@pytest.mark.parametrize("n_tied", [2000, 12000])
def test_large_tie_sets(n_tied):
    """2000 equal scores at the cut: radix over positions; 12000 equal scores:
    the level-1 bin exceeds the candidate buffer (direct pass)."""
    rng = np.random.default_rng(n_tied)
    n = 40000
    s = (rng.random((1, 2, n)) + 2.0).astype(np.float32)
    pos = rng.choice(n, n_tied, replace=False)
    s[0, :, pos] = np.float32(2.5)
    _check(s, [n], [int(np.sum(s[0, 0] < 2.5)) + n_tied // 3], 0)


def test_integer_scores_and_signed_zero():
    rng = np.random.default_rng(3)
    n = 20000
    s = rng.integers(0, 4, size=(2, 2, n)).astype(np.float32)
    s[s == 0] = np.where(rng.random(int(np.sum(s == 0))) < 0.5, np.float32(0.0), np.float32(-0.0))
    _check(s, [n, n - 3], [7000, 11111], 0)


def test_noaligned_rows():
    rng = np.random.default_rng(4)
    n = 16387                                   # rows not 16-byte aligned: scalar loads
    s = rng.random((2, 2, n)).astype(np.float32)
    _check(s, [n, 16385], [8000, 16000], 1)


@pytest.mark.parametrize("n", [8193, 40000, 70000, 90000, 110000, 125000, 131072])
def test_every_cluster_size(n):
    """1, 3, 5, 6, 7, 8 and 8 chunks per head: one cluster per KV head of that size."""
    rng = np.random.default_rng(n + 7)
    s = (rng.lognormal(0.0, 3.0, (2, 2, n))).astype(np.float32)
    lengths = [n, n - 16385 if n > 32768 else n // 2]
    s = _protect(s, lengths, 8)
    _check(s, lengths, [(n - 8) * 19 // 20, (lengths[1] - 8) // 3], 8)


def test_ties_straddle_cluster_ctas():
    """Equal scores in every chunk of a 5-chunk head, cut in the middle of them."""
    rng = np.random.default_rng(11)
    n = 80000
    s = (rng.random((1, 2, n)) + 2.0).astype(np.float32)
    s[0, :, ::7] = np.float32(2.5)
    below = int(np.sum(s[0, 0] < 2.5))
    _check(s, [n], [below + int(np.sum(s[0, 0] == 2.5)) // 2 + 3], 0)


@pytest.mark.parametrize("case", ["random", "prefix", "ties2000", "ties12000"])
def test_multi_kernel_path(case):
    """Heads longer than eight chunks use the multi-kernel radix selection."""
    rng = np.random.default_rng(5)
    n = 150000
    if case == "random":
        s = (rng.standard_normal((2, 2, n)) ** 2).astype(np.float32)
        lengths = [n, 140001]
        s = _protect(s, lengths, 8)
        _check(s, lengths, [(n - 8) * 9 // 10, 70000], 8)
        return
    s = (rng.random((1, 2, n)) + 2.0).astype(np.float32)
    if case == "prefix":
        s[0, 0, 100:140] = np.float32(2.5) + np.arange(40, dtype=np.float32) * np.float32(2 ** -22)
        _check(s, [n], [int(np.sum(s[0, 0] < 2.5)) + 17], 0)
        return
    n_tied = int(case[4:])
    pos = rng.choice(n, n_tied, replace=False)
    s[0, :, pos] = np.float32(2.5)
    _check(s, [n], [int(np.sum(s[0, 0] < 2.5)) + n_tied // 3], 0)


@pytest.mark.parametrize("n_members", [1, 200, 256, 257, 600])
def test_prefix_members_across_cluster_ctas(n_members):
    """Slots sharing the k-th item's 24-bit key prefix, spread over the CTAs
    of a 5-chunk cluster, resolved by the last digit and the tie rank.  Their
    scores differ only in the last 6 mantissa bits, with ties among them, and
    the cut falls inside them."""
    rng = np.random.default_rng(n_members + 40)
    n = 80000
    s = (rng.random((1, 2, n)) + 2.0).astype(np.float32)
    pos = rng.choice(n, n_members, replace=False)
    low = rng.integers(0, 40, size=n_members).astype(np.float32) * np.float32(2 ** -23)
    s[0][:, pos] = np.float32(1.5) + low
    below = int(np.sum(s[0, 0] < 1.5))
    _check(s, [n], [below + (n_members + 1) // 2], 0)
