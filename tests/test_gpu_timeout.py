"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes gives up after its limit (1 s), the kernel records
DROPKV_FLAG_TIMEOUT in the status word and returns, dropkv_read_status maps it
to DROPKV_ERR_TIMEOUT, and the context stays usable for the next call.

The probe kernel is compiled here from the library's own wait primitive
(csrc/sm103_ptx.cuh: mbar_wait): one thread waits on an mbarrier that no one
arrives at; another case sets the abort flag that every pipeline role polls.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, synth

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
