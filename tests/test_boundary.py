"""The C-ABI boundary: the library loads and exports what include/dropkv.h
declares (CPU), host-side validation rejects bad calls without launching, and
device-side checks report through the status word (GPU)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_dropkv_gb300 import DropKV, _binding as B, _build, synth


def test_library_exports_every_declared_symbol():
    path = _build.build_library()
    lib = ctypes.CDLL(path)
    declared = B.declared_functions()
    assert set(declared) == {"dropkv_workspace_size", "dropkv_score", "dropkv_score_timed", "dropkv_score_noalloc",
                             "dropkv_select", "dropkv_compact", "dropkv_evict", "dropkv_score_ex",
                             "dropkv_evict_ex", "dropkv_evict_prefill", "dropkv_prefill_attention", "dropkv_select_layer", "dropkv_compact_heads", "dropkv_read_status",
                             "dropkv_version"}
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if ln.split()[-1].startswith("dropkv_")})
    assert exported == declared, (exported, declared)
    lib.dropkv_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.dropkv_version()


def test_product_library_exports_no_test_hook():
    """include/dropkv_test_hooks.h is served only by the test build."""
    path = _build.build_library()
    hooks = B.declared_functions(os.path.join(_build.INCLUDE, "dropkv_test_hooks.h"))
    assert hooks == ["dropkv_test_skip_pass2_k", "dropkv_test_skip_prefill_k"]
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    assert not any(h in out for h in hooks)
    assert "DROPKV_TEST_HOOKS" not in " ".join(_build.NVCC_FLAGS)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()


def test_product_package_does_not_import_oracle():
    import kv_cache_eviction_dropkv_gb300 as pkg
    import os
    root = os.path.dirname(pkg.__file__)
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "dropkv_oracle" not in text, f


gpu = pytest.mark.gpu
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _small():
    wl = synth.make_workload("llama8b_gqa_d128_n32k", n_max=640)
    s = wl.spec
    op = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, device=DEV)
    return wl, op, wl.q.to(DEV), wl.k.to(DEV), wl.v.to(DEV), wl.lengths.to(DEV), wl.evict_k.to(DEV)


@gpu
def test_host_validation_rejects_without_launch():
    wl, op, q, k, v, lengths, ev = _small()
    s = wl.spec
    op.scores.fill_(3.0)
    call = lambda **kw: B.lib().dropkv_score(
        ctypes.byref(kw.get("shape", op.shape)), kw.get("q", B._ptr(q)), kw.get("k", B._ptr(k)), B._ptr(v),
        B._ptr(lengths), kw.get("pool", 5), kw.get("protect", 8), B._ptr(op.scores), None, B._ptr(op.workspace),
        kw.get("ws", op.workspace.numel()), B._ptr(op.status), B._stream(None))
    assert call() == 0
    torch.cuda.synchronize()
    op.scores.fill_(3.0)
    op.status.zero_()
    bad = [
        dict(pool=4), dict(pool=0), dict(pool=65), dict(protect=-1),
        dict(ws=op.workspace.numel() - 1),
        dict(q=ctypes.c_void_p(q.data_ptr() + 2)),                  # misaligned
        dict(k=None),
        dict(shape=B.make_shape(1, 32, 8, 100, 640, 8)),            # d not a multiple of 8
        dict(shape=B.make_shape(1, 30, 8, 128, 640, 8)),            # Hq % Hkv != 0
    ]
    codes = [call(**kw) for kw in bad]
    assert codes[:4] == [1, 1, 1, 1]
    assert codes[4] == 2
    assert codes[5:] == [1, 1, 6, 1]
    assert B.lib().dropkv_workspace_size(ctypes.byref(B.make_shape(1, 32, 2, 128, 640, 8))) == 0   # R = 128
    r128 = B.lib().dropkv_score(ctypes.byref(B.make_shape(1, 32, 2, 128, 640, 8)), B._ptr(q), B._ptr(k), B._ptr(v),
                                None, 5, 8, B._ptr(op.scores), None, B._ptr(op.workspace), op.workspace.numel(),
                                B._ptr(op.status), B._stream(None))
    assert r128 == 6                                              # UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(op.scores == 3.0)                            # nothing was launched
    assert int(op.status.item()) == 0
    # compact: outputs may not alias the inputs
    r = B.lib().dropkv_compact(ctypes.byref(op.shape), B._ptr(k), B._ptr(v), B._ptr(op.kept_idx),
                               B._ptr(op.kept_len), 10, B._ptr(k), B._ptr(op.v_out), B._ptr(op.status),
                               B._stream(None))
    assert r == 1
    # the one-call path checks every argument before it launches anything
    op.kept_len.fill_(-3)
    evict = lambda **kw: B.lib().dropkv_evict(
        ctypes.byref(op.shape), B._ptr(q), B._ptr(k), B._ptr(v), B._ptr(lengths), kw.get("ev", B._ptr(ev)),
        kw.get("pool", 5), 8, B._ptr(op.scores), None, B._ptr(op.kept_idx), B._ptr(op.kept_len), 10,
        kw.get("k_out", B._ptr(op.k_out)), kw.get("v_out", B._ptr(op.v_out)), B._ptr(op.workspace),
        kw.get("ws", op.workspace.numel()), B._ptr(op.status), B._stream(None))
    assert [evict(v_out=None), evict(k_out=B._ptr(k)), evict(ev=None), evict(pool=2),
            evict(ws=op.workspace.numel() - 1)] == [1, 1, 1, 1, 2]
    torch.cuda.synchronize()
    assert torch.all(op.scores == 3.0) and torch.all(op.kept_len == -3)
    assert int(op.status.item()) == 0


@gpu
def test_device_argument_flags():
    wl, op, q, k, v, lengths, ev = _small()
    s = wl.spec
    op.run(q, k, v, lengths, ev)
    assert op.check() == 0
    # eviction count beyond n_b - protect: flagged, nothing evicted
    op.reset_status()
    bad_k = torch.tensor([s.n_max - s.protect + 1], dtype=torch.int32, device=DEV)
    op.select(lengths, bad_k)
    code, flags = B.dropkv_read_status(op.status)
    assert code == 7 and flags & B.FLAG_BAD_K
    assert int(op.kept_len.item()) == s.n_max
    assert torch.equal(op.kept_idx[0, :, :s.n_max].cpu(), torch.arange(s.n_max, dtype=torch.int32).expand(s.Hkv, -1))
    # output capacity below kept_len: flagged, only out_rows rows copied
    op.reset_status()
    op.select(lengths, ev)
    small = DropKV(s.B, s.Hq, s.Hkv, s.d, s.n_max, s.w, s.pool_kernel, s.protect, out_rows=4, device=DEV)
    small.kept_idx.copy_(op.kept_idx)
    small.kept_len.copy_(op.kept_len)
    small.compact(k, v)
    code, flags = B.dropkv_read_status(small.status)
    assert code == 7 and flags & B.FLAG_OVERFLOW
    # invalid length: flagged, unit skipped
    op.reset_status()
    op.score(q, k, v, torch.tensor([3], dtype=torch.int32, device=DEV))
    code, flags = B.dropkv_read_status(op.status)
    assert code == 7 and flags & B.FLAG_BAD_LENGTH


@gpu
def test_singular_input_reported_not_patched():
    """One key more than 2000 nats above the rest: p_j is exactly 1; the oracle
    rejects it and the GPU reports SINGULAR with +inf for that slot."""
    rng = np.random.default_rng(2)
    B_, Hq, Hkv, d, n, w = 1, 2, 1, 64, 512, 2
    q = rng.standard_normal((B_, Hq, w, d)).astype(np.float32)
    k = rng.standard_normal((B_, Hkv, n, d)).astype(np.float32)
    v = rng.standard_normal((B_, Hkv, n, d)).astype(np.float32)
    q[..., 0] = 60.0
    k[0, 0, :, 0] = 0.0
    k[0, 0, 300, 0] = 300.0
    qb, kb, vb = synth.bf16_round(q), synth.bf16_round(k), synth.bf16_round(v)
    with pytest.raises(oracle.SingularInput):
        oracle.score(qb, kb, vb, np.array([n], dtype=np.int32), 1, 0)
    op = DropKV(B_, Hq, Hkv, d, n, w, 1, 0, device=DEV)
    op.score(qb.to(DEV), kb.to(DEV), vb.to(DEV), None)
    code, flags = B.dropkv_read_status(op.status)
    assert code == 3 and flags & B.FLAG_SINGULAR
    assert torch.isinf(op.raw_scores[0, 0, 300]).item()


@gpu
def test_streams_and_determinism():
    wl, op, q, k, v, lengths, ev = _small()
    op.run(q, k, v, lengths, ev)
    op.check()
    first = (op.scores.clone(), op.kept_idx.clone(), op.k_out.clone())
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        op.scores.zero_()
        op.run(q, k, v, lengths, ev, stream=st)
    op.check(st)
    assert torch.equal(first[0], op.scores)
    assert torch.equal(first[1], op.kept_idx)
    assert torch.equal(first[2].view(torch.int16), op.k_out.view(torch.int16))
