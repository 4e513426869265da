"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes gives up after its limit (1 s), the kernel records
DROPKV_FLAG_TIMEOUT in the status word and returns, dropkv_read_status maps it
to DROPKV_ERR_TIMEOUT, and the context stays usable for the next call.

The probe kernel is compiled here from the library's own wait primitive
(csrc/sm103_ptx.cuh: mbar_wait): one thread waits on an mbarrier that no one
arrives at; another case sets the abort flag that every pipeline role polls.

The pipeline cases run the real scoring call from the test build of the
library (libdropkv_test_hooks.so: 10 ms wait limit, include/dropkv_test_hooks.h),
told to leave out one K tile copy of one head: that CTA's MMA issuer gives up,
every role of the CTA leaves its loop, copies and MMAs in flight are waited
for, the tensor memory is released, the status reads DROPKV_ERR_TIMEOUT, the
other heads are scored as usual, and the next call on the same context is
clean.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import time

from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, _build, synth
from tests._parity import check_scores

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "kv_cache_eviction_dropkv_gb300",
                    "csrc")
INCLUDE = os.path.join(os.path.dirname(CSRC), "..", "include")

PROBE = r'''
#include <cuda_runtime.h>
#include <stdint.h>
#include "dropkv.h"
#include "sm103_ptx.cuh"
using namespace dropkv;
// thread 0 waits on a barrier no one arrives at; with `abort_after_ns` > 0,
// thread 32 raises the abort flag after that long instead
__global__ void wait_nothing(uint32_t* status, unsigned long long* elapsed, unsigned long long abort_after_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait(&bar, 0, &abort_flag);
    elapsed[0] = global_timer_ns() - t0;
    if (!ok) atomicOr(status, DROPKV_FLAG_TIMEOUT);
  } else if (threadIdx.x == 32 && abort_after_ns > 0) {
    const uint64_t t0 = global_timer_ns();
    uint32_t it = 0;
    while (global_timer_ns() - t0 < abort_after_ns && ++it < (1u << 30)) {
    }
    *reinterpret_cast<volatile int*>(&abort_flag) = 1;
  }
}
extern "C" int run_wait_nothing(uint32_t* status, unsigned long long* elapsed, unsigned long long abort_after_ns) {
  wait_nothing<<<1, 64>>>(status, elapsed, abort_after_ns);
  return (int)cudaDeviceSynchronize();
}
'''


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    d = tmp_path_factory.mktemp("timeout_probe")
    src = d / "probe.cu"
    src.write_text(PROBE)
    so = d / "probe.so"
    subprocess.run([shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc", "-gencode",
                    "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-I", CSRC, "-I", INCLUDE, "-o", str(so), str(src)], check=True)
    lib = ctypes.CDLL(str(so))
    lib.run_wait_nothing.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_ulonglong]
    lib.run_wait_nothing.restype = ctypes.c_int
    return lib


def _run(probe, abort_after_ns):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    assert probe.run_wait_nothing(status.data_ptr(), elapsed.data_ptr(), abort_after_ns) == 0
    code, flags = B.dropkv_read_status(status)
    return code, flags, int(elapsed.item()) / 1e9


def _context_still_works():
    wl = synth.make_workload("tiny_d16_n128", seed=42)
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    op.run(wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV), wl.lengths.to(DEV), wl.evict_k.to(DEV))
    assert op.check() == 0
    nb = int(wl.lengths[0])
    sc = op.scores.cpu().numpy()[0]
    assert np.all(np.isfinite(sc[:, :nb - s.protect])) and np.all(np.isinf(sc[:, nb - s.protect:nb]))


def test_wait_gives_up_after_its_limit(probe):
    code, flags, secs = _run(probe, 0)
    assert flags & B.FLAG_TIMEOUT and code == 8          # DROPKV_ERR_TIMEOUT
    assert 0.9 < secs < 5.0, secs                        # the 1 s limit, not a hang
    _context_still_works()


def test_wait_returns_when_another_role_aborts(probe):
    code, flags, secs = _run(probe, 50_000_000)          # abort after 50 ms
    assert flags & B.FLAG_TIMEOUT and code == 8
    assert 0.04 < secs < 0.5, secs
    _context_still_works()


@pytest.fixture(scope="module")
def hooks_lib():
    return _build.build_library(variant="test_hooks")


@pytest.mark.parametrize("case", ["dynamic_split", "dominant_split"])
def test_scoring_pipeline_times_out_and_recovers(hooks_lib, case):
    if case == "dynamic_split":
        wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=16384)
        unit, tile = 3, 40
    else:   # a sink of p ~ 0.999: unit 0's first split runs in the dominant mode
        wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=16384, sink_margin=float(np.log(999.0)))
        unit, tile = 0, 5
    s = wl.spec
    q, k, v, lengths = wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV), wl.lengths.to(DEV)
    ref = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    ref.score(q, k, v, lengths)
    assert ref.check() == 0
    want = ref.raw_scores.cpu().numpy()
    others = [h for h in range(s.Hkv) if h != unit]
    with B.use_library(hooks_lib) as L:
        assert hasattr(L, "dropkv_test_skip_pass2_k")
        op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
        assert L.dropkv_test_skip_pass2_k(unit, tile) == 0
        try:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            op.score(q, k, v, lengths)
            code, flags = B.dropkv_read_status(op.status)
            secs = time.perf_counter() - t0
        finally:
            assert L.dropkv_test_skip_pass2_k(-1, -1) == 0
        assert code == 8 and flags & B.FLAG_TIMEOUT, (code, flags)      # DROPKV_ERR_TIMEOUT
        assert secs < 0.5, secs                                        # 10 ms waits, not the 1 s of the product
        got = op.raw_scores.cpu().numpy()
        check_scores(got[:, others], want[:, others], wl.lengths.numpy(), "heads the hook left alone")
        # the same context, the hook off: a clean call, twice
        for _ in range(2):
            op.reset_status()
            op.score(q, k, v, lengths)
            assert op.check() == 0
            check_scores(op.raw_scores.cpu().numpy(), want, wl.lengths.numpy(), "call after the timeout")
    # and the product library on the same context
    ref.reset_status()
    ref.score(q, k, v, lengths)
    assert ref.check() == 0


def test_prefill_attention_times_out_and_recovers(hooks_lib):
    """The fused prefill call with one K tile copy of one KV head left out:
    every CTA of that head's query heads that reaches the tile gives up
    (10 ms waits) and raises DROPKV_FLAG_TIMEOUT, the other heads' output is
    exact, and the next calls on the same context are clean and equal the
    product library's output."""
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=2048)
    s = wl.spec
    rng = np.random.default_rng(31)
    q = torch.as_tensor(synth.bf16_round(rng.standard_normal((s.B, s.Hq, s.n_max, s.d)).astype(np.float32))).to(DEV)
    k, v, lengths, ev = wl.k.to(DEV), wl.v.to(DEV), wl.lengths.to(DEV), wl.evict_k.to(DEV)
    ref = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    out_ref = torch.empty_like(q)
    ref.run_prefill(q, k, v, lengths, ev, out_ref)
    assert ref.check() == 0
    with B.use_library(hooks_lib) as L:
        assert hasattr(L, "dropkv_test_skip_prefill_k")
        op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
        out = torch.empty_like(q)
        assert L.dropkv_test_skip_prefill_k(1, 3) == 0
        try:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            op.run_prefill(q, k, v, lengths, ev, out)
            code, flags = B.dropkv_read_status(op.status)
            secs = time.perf_counter() - t0
        finally:
            assert L.dropkv_test_skip_prefill_k(-1, -1) == 0
        # the eviction kernels after the attention also read that head's
        # window states, left unwritten, and may add their own flags (the
        # status code is the highest-precedence one): TIMEOUT must be there
        assert code != 0 and flags & B.FLAG_TIMEOUT, (code, flags)
        assert secs < 0.5, secs
        # heads of the other KV heads are computed as usual
        g = s.Hq // s.Hkv
        keep = [hq for hq in range(s.Hq) if hq // g != 1]
        assert torch.equal(out[:, keep], out_ref[:, keep])
        for _ in range(2):
            op.reset_status()
            out.zero_()
            op.run_prefill(q, k, v, lengths, ev, out)
            assert op.check() == 0
            assert torch.equal(out, out_ref)
            kl = ref.kept_len.cpu()
            assert torch.equal(op.kept_len.cpu(), kl)
            a, b_ = op.kept_idx.cpu(), ref.kept_idx.cpu()
            for b in range(s.B):
                for h in range(s.Hkv):
                    n = int(kl[b, h]) if kl.dim() == 2 else int(kl[b])
                    assert torch.equal(a[b, h, :n], b_[b, h, :n])
