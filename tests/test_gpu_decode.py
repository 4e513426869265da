"""Decode-time re-scoring on the GPU, against the oracle.

After the prefill eviction, m decode tokens are appended to the compacted
cache, the window moves to the newest w positions, and the grown cache is
scored, selected and compacted again by the same library call (the reading is
stated in kv_cache_eviction_dropkv_gb300/decode.py).  The result is compared
with the oracle run on exactly that grown cache, every output as in the other
parity tests.
"""
import numpy as np
import pytest

import oracle
from kv_cache_eviction_dropkv_gb300 import synth
from kv_cache_eviction_dropkv_gb300.decode import grow_after_eviction
from tests._gpu import DEV, _compare, _run

pytestmark = pytest.mark.gpu


def _rescore(dec, label):
    s = dec.spec
    ref = oracle.run_path(dec.q, dec.k, dec.v, dec.lengths, dec.evict_k, s.pool_kernel, s.protect)
    op, k, v, _ = _run(dec)
    _compare(dec, op, k, v, ref, label)
    return op


@pytest.mark.parametrize("m", [1, 64])
def test_rescore_after_decode_tokens_n32k(m):
    wl = synth.make_workload("llama8b_gqa_d128_n32k")
    dec = grow_after_eviction(wl, m, seed=100 + m, device=DEV)
    assert dec.spec.n_max == int(wl.kept_len()[0]) + m
    _rescore(dec, "decode m=%d" % m)


def test_rescore_after_decode_tokens_ragged_batch():
    wl = synth.make_workload("qwen_gqa7_b4_ragged_n64k", n_max=12000)
    dec = grow_after_eviction(wl, 5, seed=9, device=DEV)
    assert len(set(dec.lengths.tolist())) > 1          # still ragged
    _rescore(dec, "decode ragged")


def test_rescore_after_decode_keeps_a_sink():
    """The prefill's sink carries about 0.999 of each window row; it survives
    the prefill eviction (highest score) and, with the decode rows attending to
    it as well, survives the re-scoring too."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=8192, sink_margin=float(np.log(999.0)))
    dec = grow_after_eviction(wl, 16, seed=7, device=DEV)
    op = _rescore(dec, "decode after a sink")
    kept = op.kept_idx.cpu().numpy()
    assert np.all(kept[0, :, 0] == 0)                   # position 0 (the sink) is still kept in every head


def test_repeated_decode_steps_stay_at_budget():
    """Three re-scoring steps in a row (m = 8 each): every step evicts exactly
    m rows and matches the oracle on its own grown cache."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=6000)
    n0 = int(wl.kept_len()[0])
    for step in range(3):
        dec = grow_after_eviction(wl, 8, seed=300 + step, device=DEV)
        assert int(dec.kept_len()[0]) == n0
        _rescore(dec, "decode step %d" % step)
        wl = dec
