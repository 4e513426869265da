"""Comparison rules between the CUDA path and the oracle.

Scores: the required bound is |gpu - ref| <= 2e-3 |ref| + 1e-6 (relative error
2e-3, absolute 1e-6 for near-zero scores).  Because scores at long context are
far below 1e-6, the tests also apply a scale-aware bound
|gpu - ref| <= 2e-3 |ref| + 1e-6 * max_finite(ref of that head), which keeps
the relative test meaningful there.  +inf (protected) must match exactly.

Kept sets: they must match exactly except for tokens whose oracle score lies
within the score tolerance of the oracle's k-th smallest score (the band where
the k-th and (k+1)-th scores are indistinguishable), and the number kept must
be exact.
"""
import math

import numpy as np

RTOL = 2e-3
ATOL = 1e-6


def score_tolerance(ref_row: np.ndarray) -> np.ndarray:
    finite = np.isfinite(ref_row)
    scale = float(np.max(ref_row[finite])) if finite.any() else 0.0
    return RTOL * np.abs(ref_row) + ATOL * scale


def check_scores(got: np.ndarray, ref: np.ndarray, lengths, what: str = "scores"):
    """got/ref [B,H,n_max]; only slots j < n_b are compared.  Returns the worst
    error as a fraction of the scale-aware tolerance."""
    worst = 0.0
    B, H, _ = ref.shape
    for b in range(B):
        nb = int(lengths[b])
        for h in range(H):
            r, g = ref[b, h, :nb], got[b, h, :nb]
            inf = np.isinf(r)
            assert np.array_equal(np.isinf(g), inf), "%s: +inf slots differ (b=%d h=%d)" % (what, b, h)
            assert np.all(g[inf] == r[inf])
            fr, fg = r[~inf], g[~inf]
            assert np.all(np.isfinite(fg)), "%s: non-finite GPU score (b=%d h=%d)" % (what, b, h)
            err = np.abs(fg - fr)
            literal = RTOL * np.abs(fr) + ATOL
            assert np.all(err <= literal), "%s: literal bound violated (b=%d h=%d) max %.3g" % (
                what, b, h, float(np.max(err / literal)))
            tol = score_tolerance(r)[~inf]
            frac = err / np.where(tol > 0, tol, 1e-300)
            if frac.size:
                worst = max(worst, float(frac.max()))
            assert np.all(err <= tol), "%s: scale-aware bound violated (b=%d h=%d) worst %.3g of tol" % (
                what, b, h, float(frac.max()))
    return worst


def check_kept(kept_gpu: np.ndarray, len_gpu: np.ndarray, kept_ref: np.ndarray, len_ref: np.ndarray,
               final_ref: np.ndarray, lengths, evict_k):
    """Exact kept sets outside the tolerance band around the k-th smallest score."""
    assert np.array_equal(len_gpu, len_ref), (len_gpu, len_ref)
    B, H, _ = final_ref.shape
    band_total = 0
    for b in range(B):
        nb, kb, kl = int(lengths[b]), int(evict_k[b]), int(len_ref[b])
        for h in range(H):
            g = kept_gpu[b, h, :kl]
            assert np.all(np.diff(g) > 0), "kept indices must be strictly ascending (b=%d h=%d)" % (b, h)
            assert g.min() >= 0 and g.max() < nb
            r = kept_ref[b, h, :kl]
            if np.array_equal(g, r):
                continue
            fin = final_ref[b, h, :nb]
            if kb == 0:
                raise AssertionError("nothing to evict but kept sets differ (b=%d h=%d)" % (b, h))
            order = np.lexsort((np.arange(nb), fin))
            T = fin[order[kb - 1]]
            tolT = RTOL * abs(T) + ATOL * float(np.max(fin[np.isfinite(fin)]))
            band = np.abs(fin - T) <= tolT
            diff = np.setxor1d(g, r)
            assert np.all(band[diff]), "kept sets differ outside the tolerance band (b=%d h=%d): %s" % (
                b, h, diff[~band[diff]][:10])
            band_total += diff.size
    return band_total


def check_kept_layer(kept_gpu, len_gpu, kept_ref, len_ref, final_ref, lengths, evict_total):
    """Layer-wide selection: per sequence, the kept set (over all heads) must
    match the oracle's except for slots whose oracle score lies within the
    tolerance of the pool's evict_total-th smallest score; the total kept per
    sequence must be exact.  kept_*: [B,H,n_max], len_*: [B,H]."""
    B, H, _ = final_ref.shape
    band_total = 0
    for b in range(B):
        nb, e = int(lengths[b]), int(evict_total[b])
        assert int(len_gpu[b].sum()) == int(len_ref[b].sum()) == H * nb - e
        got = np.zeros((H, nb), dtype=bool)
        ref = np.zeros((H, nb), dtype=bool)
        for h in range(H):
            g = kept_gpu[b, h, :len_gpu[b, h]]
            assert np.all(np.diff(g) > 0), "kept indices must be strictly ascending (b=%d h=%d)" % (b, h)
            if g.size:
                assert g.min() >= 0 and g.max() < nb
            got[h, g] = True
            ref[h, kept_ref[b, h, :len_ref[b, h]]] = True
        if np.array_equal(got, ref):
            continue
        fin = final_ref[b, :, :nb]
        assert e > 0, "nothing to evict but kept sets differ (b=%d)" % b
        flat = fin.reshape(-1)
        T = flat[np.lexsort((np.arange(flat.size), flat))[e - 1]]
        tolT = RTOL * abs(T) + ATOL * float(np.max(flat[np.isfinite(flat)]))
        band = np.abs(fin - T) <= tolT
        diff = got != ref
        assert np.all(band[diff]), "kept sets differ outside the tolerance band (b=%d)" % b
        band_total += int(diff.sum())
    return band_total


def deletion_score(q, k, v, lengths, j=0):
    """Raw score of key j by deletion, in fp64 (the pages' definition of the
    perturbation: Delta_j = a_{-j} - a = p_j (a_{-j} - v_j), "DropKV: Exact
    single-entry output-perturbation scoring", Core equation): a_{-j} is the
    softmax output over the other keys and 1 - p_j their mass, both summed
    directly, so nothing cancels however close p_j is to 1.  q, k, v are float64
    arrays [B,Hq,w,d] / [B,Hkv,n,d]; returns [B,Hkv]."""
    B, Hq, w, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hkv))
    for b in range(B):
        nb = int(lengths[b])
        for h in range(Hkv):
            acc = 0.0
            for hl in range(g):
                for t in range(w):
                    pos = nb - w + t
                    if j > pos:
                        continue
                    qq = q[b, h * g + hl, t]
                    x = k[b, h, :pos + 1] @ qq / math.sqrt(d)
                    others = np.arange(pos + 1) != j
                    xr = x[others]
                    if xr.size == 0:
                        return None                        # a single visible key: removal is singular
                    mr = xr.max()
                    er = np.exp(xr - mr)
                    a_rest = er @ v[b, h, :pos + 1][others] / er.sum()
                    rest = np.exp(mr - x[j]) * er.sum()     # (1 - p_j) / p_j
                    pj = 1.0 / (1.0 + rest)
                    acc += pj * pj * float(((a_rest - v[b, h, j]) ** 2).sum())
            out[b, h] = acc / g
    return out
