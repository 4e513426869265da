"""The scorer fused into the prompt's prefill attention (dropkv_evict_prefill).

One kernel computes the causal attention of every query row ("DropKV:
Decoupling ...", section 2.1); its last w rows are step S1's window rows, so
the eviction runs without pass 1.  Checked against the oracle:
 - the attention output of every row (oracle.prefill_attention), within the
   error of bf16 P and a bf16 output: |gpu - ref| <= 2^-8 (|ref| + max|v|);
 - the window statistics (lse, a) against S1 of the oracle on the window rows,
   at the bounds of the other parity tests;
 - the scores, kept sets and compaction against oracle.run_path on the window
   rows, exactly as every other parity test (tests/_gpu.py: _compare).
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, synth
from tests._gpu import DEV, SENTINEL, _compare

pytestmark = pytest.mark.gpu


def _prefill_inputs(wl, seed):
    """Every query row: seeded N(0, 1) bf16 rows, with the workload's own
    window rows at positions n_b - w .. n_b - 1 of each sequence (so its sink
    and needles keep their meaning)."""
    s = wl.spec
    rng = np.random.default_rng(seed)
    q = synth.bf16_round(rng.standard_normal((s.B, s.Hq, s.n_max, s.d)).astype(np.float32))
    for b in range(s.B):
        nb = int(wl.lengths[b])
        q[b, :, nb - s.w:nb] = wl.q[b]
    return q


def _window_q(q, lengths, w):
    return torch.stack([q[b, :, int(lengths[b]) - w:int(lengths[b])] for b in range(q.shape[0])]).contiguous()


def _run_prefill(wl, q_full, poison=True):
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    k, v = wl.k.clone(), wl.v.clone()
    if poison:
        for b in range(s.B):
            nb = int(wl.lengths[b])
            k[b, :, nb:] = float("nan")
            v[b, :, nb:] = float("nan")
    q, k, v = q_full.to(DEV), k.to(DEV), v.to(DEV)
    out = torch.full((s.B, s.Hq, s.n_max, s.d), -3.5, dtype=torch.bfloat16, device=DEV)
    op.scores.fill_(SENTINEL)
    op.raw_scores.fill_(SENTINEL)
    op.kept_idx.fill_(-5)
    op.run_prefill(q, k, v, wl.lengths.to(DEV), wl.evict_k.to(DEV), out)
    op.check()
    return op, k, v, out


def _check_output(out, ref, v, lengths, g, rows=None, label=""):
    """|gpu - ref| <= 2^-8 (|ref| + max_j |v_j|) on every written row; rows past
    n_b untouched."""
    got = out.float().cpu().numpy()
    B, Hq = got.shape[:2]
    for b in range(B):
        nb = int(lengths[b])
        hi = nb if rows is None else min(nb, rows)
        for hq in range(Hq):
            vmax = float(np.abs(v[b, hq // g, :nb].float().numpy()).max())
            err = np.abs(got[b, hq, :hi] - ref[b, hq, :hi])
            tol = 2.0 ** -8 * (np.abs(ref[b, hq, :hi]) + vmax)
            assert np.all(err <= tol), "%s b=%d hq=%d: worst %.3g of the bound" % (label, b, hq, (err / tol).max())
        if rows is None:
            assert np.all(got[b, :, nb:] == -3.5), "rows past n_b were written"


def _check_path(wl, q_full, label):
    s = wl.spec
    op, k, v, out = _run_prefill(wl, q_full)
    qw = _window_q(q_full, wl.lengths, s.w)
    win = synth.Workload(spec=s, q=qw, k=wl.k, v=wl.v, lengths=wl.lengths, evict_k=wl.evict_k)
    ref = oracle.run_path(qw, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect)
    _compare(win, op, k, v, ref, label)
    return op, out


@pytest.mark.parametrize("case", ["gqa_ragged", "mha_d96", "tiny_d16"])
def test_prefill_output_and_eviction_vs_oracle(case):
    if case == "gqa_ragged":
        wl = synth.make_workload("qwen_gqa7_b4_ragged_n64k", n_max=900)
    elif case == "mha_d96":
        wl = synth.make_workload("phi3mini_mha_d96_n4k", n_max=600)
    else:
        wl = synth.make_workload("tiny_d16_n128", seed=43)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=11)
    op, out = _check_path(wl, q_full, "prefill " + case)
    ref_out = oracle.prefill_attention(q_full, wl.k, wl.v, wl.lengths.numpy())
    _check_output(out, ref_out, wl.v, wl.lengths.numpy(), s.g, label=case)


@pytest.mark.parametrize("n", [1000, 1030, 1153])
def test_prefill_tile_pairing_edges(n):
    """The CTA tiling's edge cases on a GQA layer: n = 1000 leaves an odd
    number of tiles before the window (the last pair CTA has one tile), n =
    1030 puts the window across two query tiles (two window tiles, the first
    full), n = 1153 leaves one row in the last tile.  Every row's output and
    the eviction against the oracle."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=n)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=19)
    op, out = _check_path(wl, q_full, "prefill pairing n=%d" % n)
    ref_out = oracle.prefill_attention(q_full, wl.k, wl.v, wl.lengths.numpy())
    _check_output(out, ref_out, wl.v, wl.lengths.numpy(), s.g, label="pairing n=%d" % n)


def test_prefill_leaves_rows_past_each_sequence_untouched():
    """A ragged batch at a longer n_max, called twice (the second time with
    shorter lengths): no call writes an output row at or past its sequence's
    length."""
    wl = synth.make_workload("qwen_gqa7_b4_ragged_n64k", n_max=5000)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=20)
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    q, k, v = q_full.to(DEV), wl.k.to(DEV), wl.v.to(DEV)
    out = torch.full((s.B, s.Hq, s.n_max, s.d), -3.5, dtype=torch.bfloat16, device=DEV)
    for lengths in (wl.lengths, torch.clamp(wl.lengths - 150, min=s.w + s.protect + int(wl.evict_k.max()) + 1)):
        out.fill_(-3.5)
        op.run_prefill(q, k, v, lengths.to(torch.int32).to(DEV), wl.evict_k.to(DEV), out)
        op.check()
        got = out.float().cpu().numpy()
        for b in range(s.B):
            nb = int(lengths[b])
            assert np.all(got[b, :, nb:] == -3.5), "b=%d: rows past n_b = %d written (first at %s)" % (
                b, nb, np.argwhere(got[b, :, nb:] != -3.5)[:1].tolist())
            miss = np.argwhere(np.all(got[b, :, :nb] == -3.5, axis=-1))
            assert len(miss) == 0, "b=%d (n_b = %d): %d rows not written, e.g. (head, row) %s; query tiles %s" % (
                b, nb, len(miss), miss[:6].tolist(), sorted(set((miss[:, 1] // 128).tolist()))[:20])


def _prefill_sweep_cases(count, seed):
    """Random shapes for the prefill path: d, g, w up to g w = 64, ragged
    lengths, every pooling size and protection width."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < count:
        Hkv = int(rng.integers(1, 3))
        g = int(rng.integers(1, 9))
        w = int(rng.integers(1, 9))
        if g * w > 64:
            continue
        d = int(rng.choice([8, 16, 24, 64, 96, 120, 128]))
        B = int(rng.integers(1, 4))
        n = int(rng.integers(w + 1, 1400))
        lens = rng.integers(max(w, 1), n + 1, size=B)
        protect = int(rng.integers(0, w + 1))
        pool = int(rng.choice([1, 3, 5, 9]))
        evict = [int(rng.integers(0, max(1, int(L) - protect) + 1)) for L in lens]
        cases.append((B, g * Hkv, Hkv, d, n, w, pool, protect, lens.tolist(), evict))
    return cases


@pytest.mark.parametrize("case", _prefill_sweep_cases(8, 2027))
def test_prefill_random_shape_sweep(case):
    """The fused prefill on random shapes: every row's output and the whole
    eviction against the oracle, as the fixed cases above."""
    B, Hq, Hkv, d, n, w, pool, protect, lens, evict = case
    rng = np.random.default_rng(sum(lens) + d + 7)
    q_full = synth.bf16_round(rng.standard_normal((B, Hq, n, d)).astype(np.float32))
    k = synth.bf16_round(rng.standard_normal((B, Hkv, n, d)).astype(np.float32))
    v = synth.bf16_round(rng.standard_normal((B, Hkv, n, d)).astype(np.float32))
    lengths = torch.tensor(lens, dtype=torch.int32)
    spec = synth.WorkloadSpec("custom", B, Hq, Hkv, d, n, w, pool, protect, 0, "custom")
    wl = synth.Workload(spec=spec, q=_window_q(q_full, lengths, w), k=k, v=v, lengths=lengths,
                        evict_k=torch.tensor(evict, dtype=torch.int32))
    op, out = _check_path(wl, q_full, "prefill sweep %s" % (case,))
    ref_out = oracle.prefill_attention(q_full, k, v, lengths.numpy())
    _check_output(out, ref_out, v, lengths.numpy(), Hq // Hkv, label="sweep %s" % (case,))


def test_prefill_full_size_c1_layer():
    """The Phi-3-like MHA layer at its full size (n = 4096, 32 heads): every
    row's output and the whole eviction against the oracle."""
    wl = synth.make_workload("phi3mini_mha_d96_n4k")
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=12)
    op, out = _check_path(wl, q_full, "prefill n4k")
    ref_out = oracle.prefill_attention(q_full, wl.k, wl.v, wl.lengths.numpy())
    _check_output(out, ref_out, wl.v, wl.lengths.numpy(), s.g, label="n4k")


def test_prefill_full_size_n32k():
    """n = 32K, GQA 4: the eviction against the oracle in full; the output on
    the first 1024 rows (causal: they depend only on the first 1024 keys, so
    the oracle runs on that prefix)."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k")
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=13)
    op, out = _check_path(wl, q_full, "prefill n32k")
    P = 1024
    ref_out = oracle.prefill_attention(q_full[:, :, :P].contiguous(), wl.k[:, :, :P].contiguous(),
                                       wl.v[:, :, :P].contiguous())
    _check_output(out[:, :, :P], ref_out, wl.v[:, :, :P], np.full(s.B, P), s.g, rows=P, label="n32k prefix")


def test_prefill_with_dominated_rows():
    """A sink carrying 0.999 of each window row: the window state is one
    partial per row, so the dominated heads are scored in the dominant mode
    over all of their tiles by one CTA; exact against the oracle."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=5000, sink_margin=float(np.log(999.0)))
    q_full = _prefill_inputs(wl, seed=14)
    _check_path(wl, q_full, "prefill sink")


def test_prefill_with_value_offset_and_sink():
    """Values sharing an 8-sigma offset (the expanded distance's hard case)
    and a sink of about 0.9999 of each window row's mass, through the fused
    call: the window states of one partial per row take the shifted basis and
    the dominant mode; exact against the oracle, and every row's output."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=3000, sink_margin=float(np.log(9999.0)), v_offset=8.0)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=21)
    op, out = _check_path(wl, q_full, "prefill offset + sink")
    ref_out = oracle.prefill_attention(q_full, wl.k, wl.v, wl.lengths.numpy())
    _check_output(out, ref_out, wl.v, wl.lengths.numpy(), s.g, label="offset + sink")


def test_prefill_matches_the_window_path():
    """The same layer through dropkv_evict (pass 1 over the window rows) and
    through the prefilled call: scores within the tolerance of each other and
    the same kept count."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=3000)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=15)
    op_pf, _, _, _ = _run_prefill(wl, q_full, poison=False)
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    op.run(_window_q(q_full, wl.lengths, s.w).to(DEV), wl.k.to(DEV), wl.v.to(DEV), wl.lengths.to(DEV),
           wl.evict_k.to(DEV))
    op.check()
    a, b = op.raw_scores.cpu().numpy(), op_pf.raw_scores.cpu().numpy()
    scale = np.abs(a).max(axis=-1, keepdims=True)
    assert np.all(np.abs(a - b) <= 2e-3 * np.abs(a) + 1e-6 * scale)
    assert np.array_equal(op.kept_len.cpu().numpy(), op_pf.kept_len.cpu().numpy())


def test_attention_alone_equals_the_fused_output():
    """dropkv_prefill_attention runs the fused call's kernel without the
    eviction: the same bytes."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=1500)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=16)
    op, k, v, out = _run_prefill(wl, q_full, poison=False)
    out2 = torch.full_like(out, -3.5)
    op.prefill_attention(q_full.to(DEV), k, v, wl.lengths.to(DEV), out2)
    op.check()
    assert torch.equal(out, out2)


def test_prefill_snapkv_kind_vs_oracle():
    """The SnapKV score kind through the fused call (K only in pass 2; the
    window states still come from the prefill attention)."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=2500)
    s = wl.spec
    q_full = _prefill_inputs(wl, seed=17)
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV, kind="snapkv")
    k, v = wl.k.to(DEV), wl.v.to(DEV)
    out = torch.empty((s.B, s.Hq, s.n_max, s.d), dtype=torch.bfloat16, device=DEV)
    op.scores.fill_(SENTINEL)
    op.raw_scores.fill_(SENTINEL)
    op.kept_idx.fill_(-5)
    op.run_prefill(q_full.to(DEV), k, v, wl.lengths.to(DEV), wl.evict_k.to(DEV), out)
    op.check()
    qw = _window_q(q_full, wl.lengths, s.w)
    win = synth.Workload(spec=s, q=qw, k=wl.k, v=wl.v, lengths=wl.lengths, evict_k=wl.evict_k)
    ref = oracle.run_path(qw, wl.k, wl.v, wl.lengths, wl.evict_k, s.pool_kernel, s.protect, kind="snapkv")
    _compare(win, op, k, v, ref, "prefill snapkv", kind="snapkv")


def test_prefill_entry_points_reject_bad_arguments():
    """Host checks of dropkv_evict_prefill and dropkv_prefill_attention: an
    output overlapping q, k or v, a misaligned pointer or a short workspace is
    rejected with nothing launched."""
    import ctypes
    from kv_cache_eviction_dropkv_gb300 import _binding as B
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=700)
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    q = _prefill_inputs(wl, seed=18).to(DEV)
    k, v = wl.k.to(DEV), wl.v.to(DEV)
    out = torch.full_like(q, -3.5)
    L = B.lib()

    def attn(o=None, qq=None, ws=None):
        return L.dropkv_prefill_attention(ctypes.byref(op.shape), qq or B._ptr(q), B._ptr(k), B._ptr(v), None,
                                          o or B._ptr(out), B._ptr(op.workspace),
                                          op.workspace.numel() if ws is None else ws, B._ptr(op.status),
                                          B._stream(None))
    assert attn(o=B._ptr(q)) == 1                                          # output on top of q
    assert attn(o=ctypes.c_void_p(k.data_ptr())) == 1                      # ... or of k
    assert attn(qq=ctypes.c_void_p(q.data_ptr() + 2)) == 1                 # misaligned
    assert attn(ws=1024) == 2                                              # workspace too small
    fused = L.dropkv_evict_prefill(ctypes.byref(op.shape), 0, B._ptr(q), B._ptr(k), B._ptr(v), None,
                                   B._ptr(wl.evict_k.to(DEV)), 5, 8, B._ptr(q), B._ptr(op.scores), None,
                                   B._ptr(op.kept_idx), B._ptr(op.kept_len), op.out_rows, B._ptr(op.k_out),
                                   B._ptr(op.v_out), B._ptr(op.workspace), op.workspace.numel(), B._ptr(op.status),
                                   B._stream(None))
    assert fused == 1
    torch.cuda.synchronize()
    assert torch.all(out == -3.5) and int(op.status.item()) == 0           # nothing was launched
    assert attn() == 0
    op.check()
    assert not torch.all(out == -3.5)
