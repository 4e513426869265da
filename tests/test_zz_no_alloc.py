"""dropkv_score_noalloc: scoring for callers that cannot allocate device
memory when they score (a host framework that owns all device memory through
its own pool, or a serving loop that forbids allocations after start-up).

Checked through the C ABI against dropkv_score on the same inputs, with the
tolerance of the other parity tests, on two calls in a row.  Before those
calls the shared scratch array is left holding other contents (a call on a
different, single-sequence shape, and a call on NaN inputs), so a value the
entry point read before writing would show up.  Also: the oracle agrees, the
device's free memory does not change across calls, and overlapping score
buffers are rejected.  This file is collected last so that a run stopping at
the first failure has run every other test first; it also passes on its own in
a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth
from tests._parity import check_scores

pytestmark = pytest.mark.gpu

SENTINEL = -7.25


def _noalloc(shape, q, k, v, lengths, pool, protect, like_scores):
    scores = torch.full_like(like_scores, SENTINEL)
    raw = torch.full_like(like_scores, SENTINEL)
    status = torch.zeros(1, dtype=torch.int32, device=like_scores.device)
    B.dropkv_score_noalloc(shape, q, k, v, lengths, pool, protect, scores, raw, status)
    code, flags = B.dropkv_read_status(status)
    return scores, raw, code, flags


def _leave_other_contents(dev):
    """Run the entry point on another shape and on NaN inputs, so the scratch
    array holds values unrelated to the next call."""
    other = synth.make_workload("llama8b_gqa_d128_n32k", n_max=5000, seed=77)
    s = other.spec
    shape = B.make_shape(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w)
    like = torch.empty(s.B, s.Hkv, s.n_max, dtype=torch.float32, device=dev)
    q, k, v = other.q.to(dev), other.k.to(dev), other.v.to(dev)
    _noalloc(shape, q, k, v, None, s.pool_kernel, s.protect, like)
    nan = torch.full_like(k, float("nan"))
    _, _, code, _ = _noalloc(shape, torch.full_like(q, float("nan")), nan, nan, None, s.pool_kernel, s.protect, like)
    assert code != 0          # NaN inputs are reported, not silently scored


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = torch.device("cuda", 0)
    wl = synth.make_workload("qwen_gqa7_b4_ragged_n64k", n_max=9000)   # ragged, several tiles per CTA
    s = wl.spec
    lengths_np = wl.lengths.numpy()
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=dev)
    q, k, v, lengths = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev), wl.lengths.to(dev)
    op.score(q, k, v, lengths)
    assert op.check() == 0
    ref_final = op.scores.cpu().numpy()
    ref_raw = op.raw_scores.cpu().numpy()
    _leave_other_contents(dev)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(dev)[0]
    for call in range(2):
        scores, raw, code, flags = _noalloc(op.shape, q, k, v, lengths, s.pool_kernel, s.protect, op.scores)
        assert code == 0, "call %d: status %d flags 0x%x" % (call, code, flags)
        got_final, got_raw = scores.cpu().numpy(), raw.cpu().numpy()
        check_scores(got_final, ref_final, lengths_np, "noalloc call %d final" % call)
        check_scores(got_raw, ref_raw, lengths_np, "noalloc call %d raw" % call)
        for b in range(s.B):
            nb = int(lengths_np[b])
            assert np.all(got_final[b, :, nb:] == SENTINEL) and np.all(got_raw[b, :, nb:] == SENTINEL)
        del scores, raw
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    # nothing was allocated on the device by the calls (torch's own cache is emptied)
    assert torch.cuda.mem_get_info(dev)[0] >= free0


def test_noalloc_matches_the_oracle():
    dev = torch.device("cuda", 0)
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=4096 + 77)
    s = wl.spec
    ref = oracle.score(wl.q, wl.k, wl.v, wl.lengths.numpy(), s.pool_kernel, s.protect)
    shape = B.make_shape(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w)
    like = torch.empty(s.B, s.Hkv, s.n_max, dtype=torch.float32, device=dev)
    scores, raw, code, _ = _noalloc(shape, wl.q.to(dev), wl.k.to(dev), wl.v.to(dev), wl.lengths.to(dev),
                                    s.pool_kernel, s.protect, like)
    assert code == 0
    check_scores(raw.cpu().numpy(), ref["raw"], wl.lengths.numpy(), "noalloc raw vs oracle")
    check_scores(scores.cpu().numpy(), ref["final"], wl.lengths.numpy(), "noalloc final vs oracle")


def test_noalloc_rejects_overlapping_score_buffers():
    dev = torch.device("cuda", 0)
    shape = B.make_shape(1, 4, 2, 64, 1000, 4)
    q = torch.zeros(1, 4, 4, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 2, 1000, 64, dtype=torch.bfloat16, device=dev)
    buf = torch.zeros(2 * 1000 + 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(B.DropKVError) as e:
        B.dropkv_score_noalloc(shape, q, k, k, None, 3, 4, buf[:2000], buf[16:2016], status)
    assert e.value.code == 1                                 # DROPKV_ERR_INVALID_ARG, nothing launched
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda", 0)
    big = B.make_shape(8, 64, 8, 128, 131072, 8)          # scoring scratch far above 16 MiB
    t = torch.zeros(64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(B.DropKVError) as e:
        B.dropkv_score_noalloc(big, t, t, t, None, 5, 8, t, None, status)
    assert e.value.code == 2                                 # DROPKV_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert int(status.item()) == 0
