"""dropkv_score_noalloc: scoring for callers that cannot allocate device
memory when they score (a host framework that owns all device memory through
its own pool, or a serving loop that forbids allocations after start-up).

Checked through the C ABI against dropkv_score on the same inputs, on two
calls in a row (the second call sees the first call's leftovers in the shared
scratch array), with the tolerance of the other parity tests.  This file is
collected last so that a run stopping at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth
from tests._parity import check_scores

pytestmark = pytest.mark.gpu

SENTINEL = -7.25


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
    for call in range(2):
        scores = torch.full_like(op.scores, SENTINEL)
        raw = torch.full_like(op.raw_scores, SENTINEL)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        B.dropkv_score_noalloc(op.shape, q, k, v, lengths, s.pool_kernel, s.protect, scores, raw, status)
        code, flags = B.dropkv_read_status(status)
        assert code == 0, "call %d: status %d flags 0x%x" % (call, code, flags)
        got_final, got_raw = scores.cpu().numpy(), raw.cpu().numpy()
        check_scores(got_final, ref_final, lengths_np, "noalloc call %d final" % call)
        check_scores(got_raw, ref_raw, lengths_np, "noalloc call %d raw" % call)
        for b in range(s.B):
            nb = int(lengths_np[b])
            assert np.all(got_final[b, :, nb:] == SENTINEL) and np.all(got_raw[b, :, nb:] == SENTINEL)


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
