"""CPU oracle for the DropKV scoring path.  TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (dropkv_oracle.c) behind a ctypes wrapper.  Only
the test suite, the smoke check and the benchmark's CPU-baseline leg may import
it; the product package never does, and the two share no code.  The oracle is
pinned to the pages and to the mathematics by the `-m "not gpu"` tests
(brute-force deletion, library routines, invariants, the approximation bound).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dropkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libdropkv_oracle.so")

OK, INVALID, SINGULAR, NOMEM = 0, 1, 3, 9
_F64, _BF16 = 0, 1

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


class SingularInput(OracleError):
    """Some p_j equals 1: exact removal of key j is singular and is rejected."""


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    hdr = os.path.join(_HERE, "dropkv_oracle.h")
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB)
    return _LIB


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n_max", ctypes.c_int32), ("w", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_score.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, P, P, P, P,
                                         ctypes.c_int, ctypes.c_int, P, P, P, P, P, ctypes.c_int, P]
            lib.oracle_score.restype = ctypes.c_int
            lib.oracle_score_kind.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, ctypes.c_int, P, P, P, P,
                                              ctypes.c_int, ctypes.c_int, P, P, P, P, P, ctypes.c_int, P]
            lib.oracle_score_kind.restype = ctypes.c_int
            lib.oracle_select.argtypes = [ctypes.POINTER(_Shape), P, P, P, ctypes.c_int, P, P]
            lib.oracle_select.restype = ctypes.c_int
            lib.oracle_compact.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, P, P, P, P,
                                           ctypes.c_int, P, P]
            lib.oracle_compact.restype = ctypes.c_int
            lib.oracle_select_layer.argtypes = [ctypes.POINTER(_Shape), P, P, P, ctypes.c_int, P, P]
            lib.oracle_select_layer.restype = ctypes.c_int
            lib.oracle_compact_heads.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, P, P, P, P,
                                                 ctypes.c_int, P, P]
            lib.oracle_compact_heads.restype = ctypes.c_int
            lib.oracle_prefill_attention.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, P, P, P, P, P,
                                                     ctypes.c_int]
            lib.oracle_prefill_attention.restype = ctypes.c_int
            _lib = lib
    return _lib


class use_library:
    """Temporarily route the wrapper to another build of the oracle (the pin
    tests use it to check that planted mistakes are caught)."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_score", "oracle_score_kind", "oracle_select", "oracle_compact", "oracle_select_layer",
                     "oracle_compact_heads"):
            getattr(lib, name).argtypes = getattr(self.saved, name).argtypes
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source to out_path (tests only)."""
    d = os.path.dirname(out_path)
    csrc = os.path.join(d, "variant.c")
    with open(csrc, "w") as f:
        f.write(source_text)
    import shutil
    shutil.copy(os.path.join(_HERE, "dropkv_oracle.h"), os.path.join(d, "dropkv_oracle.h"))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-o", out_path, csrc, "-lm"], check=True, cwd=d)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_input(x):
    """torch bf16 tensor -> uint16 bit patterns; anything else -> contiguous float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                            .view(np.uint16)), _BF16
            x = x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.float64), _F64


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


KINDS = {"dropkv": 0, "snapkv": 1}


def score(q, k, v, lengths=None, pool_kernel: int = 1, protect: int = 0,
          nthreads: Optional[int] = None, want_stats: bool = True, kind: str = "dropkv") -> dict:
    """Run steps S1-S5.  q [B,Hq,w,d]; k, v [B,Hkv,n_max,d]; lengths [B] (None: n_max).

    Returns dict with m, l [B,Hq,w], a [B,Hq,w,d] (if want_stats), raw and final
    [B,Hkv,n_max] (NaN beyond n_b).  Raises SingularInput for p_j == 1 (DropKV
    kind only).  kind "snapkv" scores each key by the window sum of its
    attention probabilities instead of the perturbation."""
    qa, dt_q = _as_input(q)
    ka, dt_k = _as_input(k)
    va, dt_v = _as_input(v)
    if not (dt_q == dt_k == dt_v):
        raise OracleError("q, k, v must share one element type")
    B, Hq, w, d = qa.shape
    _, Hkv, n_max, _ = ka.shape
    if lengths is None:
        lens = np.full(B, n_max, dtype=np.int32)
    else:
        lens = np.ascontiguousarray(np.asarray(lengths), dtype=np.int32)
    shape = _Shape(B, Hq, Hkv, d, n_max, w)
    m = np.empty((B, Hq, w)) if want_stats else None
    l = np.empty((B, Hq, w)) if want_stats else None
    a = np.empty((B, Hq, w, d)) if want_stats else None
    raw = np.empty((B, Hkv, n_max))
    fin = np.empty((B, Hkv, n_max))
    su = np.zeros(1, dtype=np.int32)
    nt = nthreads if nthreads is not None else default_threads()
    st = _load().oracle_score_kind(ctypes.byref(shape), KINDS[kind], dt_q, _ptr(qa), _ptr(ka), _ptr(va),
                                   _ptr(lens), pool_kernel, protect,
                                   _ptr(m) if want_stats else None, _ptr(l) if want_stats else None,
                                   _ptr(a) if want_stats else None, _ptr(raw), _ptr(fin), nt, _ptr(su))
    if st == SINGULAR:
        raise SingularInput("p_j == 1 in unit %d" % int(su[0]))
    if st != OK:
        raise OracleError("oracle_score failed with status %d" % st)
    return {"m": m, "l": l, "a": a, "raw": raw, "final": fin}


def prefill_attention(q, k, v, lengths=None, nthreads: Optional[int] = None) -> np.ndarray:
    """Causal prefill attention of every query row: q [B,Hq,n_max,d], k, v
    [B,Hkv,n_max,d] -> out [B,Hq,n_max,d] float64 (NaN for rows >= n_b)."""
    qa, dt_q = _as_input(q)
    ka, dt_k = _as_input(k)
    va, dt_v = _as_input(v)
    if not (dt_q == dt_k == dt_v):
        raise OracleError("q, k, v must share one element type")
    B, Hq, n_max, d = qa.shape
    Hkv = ka.shape[1]
    lens = (np.full(B, n_max, dtype=np.int32) if lengths is None
            else np.ascontiguousarray(np.asarray(lengths), dtype=np.int32))
    out = np.empty((B, Hq, n_max, d))
    shape = _Shape(B, Hq, Hkv, d, n_max, 1)
    st = _load().oracle_prefill_attention(ctypes.byref(shape), dt_q, _ptr(qa), _ptr(ka), _ptr(va), _ptr(lens),
                                          _ptr(out), nthreads if nthreads is not None else default_threads())
    if st != OK:
        raise OracleError("oracle_prefill_attention failed with status %d" % st)
    return out


def select(final, lengths, evict_k, protect: int = 0):
    """Step S6.  Returns (kept_idx [B,Hkv,n_max] int32, first kept_len[b] valid; kept_len [B])."""
    fin = np.ascontiguousarray(final, dtype=np.float64)
    B, Hkv, n_max = fin.shape
    lens = np.ascontiguousarray(np.asarray(lengths), dtype=np.int32)
    ks = np.ascontiguousarray(np.asarray(evict_k), dtype=np.int32)
    kept = np.full((B, Hkv, n_max), -1, dtype=np.int32)
    kl = np.zeros(B, dtype=np.int32)
    shape = _Shape(B, Hkv, Hkv, 1, n_max, 1)
    st = _load().oracle_select(ctypes.byref(shape), _ptr(fin), _ptr(lens), _ptr(ks), protect,
                               _ptr(kept), _ptr(kl))
    if st != OK:
        raise OracleError("oracle_select failed with status %d" % st)
    return kept, kl


def select_layer(final, lengths, evict_total, protect: int = 0):
    """Layer-wide bottom-k (AdaDropKV): per sequence, evict the evict_total[b]
    smallest (score, head, position) over all KV heads.  Returns (kept_idx
    [B,Hkv,n_max] int32, first kept_len[b,h] valid; kept_len [B,Hkv])."""
    fin = np.ascontiguousarray(final, dtype=np.float64)
    B, Hkv, n_max = fin.shape
    lens = np.ascontiguousarray(np.asarray(lengths), dtype=np.int32)
    et = np.ascontiguousarray(np.asarray(evict_total), dtype=np.int32)
    kept = np.full((B, Hkv, n_max), -1, dtype=np.int32)
    kl = np.zeros((B, Hkv), dtype=np.int32)
    shape = _Shape(B, Hkv, Hkv, 1, n_max, 1)
    st = _load().oracle_select_layer(ctypes.byref(shape), _ptr(fin), _ptr(lens), _ptr(et), protect,
                                     _ptr(kept), _ptr(kl))
    if st != OK:
        raise OracleError("oracle_select_layer failed with status %d" % st)
    return kept, kl


def compact_heads(k, v, kept_idx, kept_len, out_rows: int):
    """Gather with a kept count per KV head (kept_len [B,Hkv])."""
    ka = np.ascontiguousarray(k)
    va = np.ascontiguousarray(v)
    B, Hkv, n_max, d = ka.shape
    idx = np.ascontiguousarray(kept_idx, dtype=np.int32)
    kl = np.ascontiguousarray(kept_len, dtype=np.int32)
    k_out = np.zeros((B, Hkv, out_rows, d), dtype=ka.dtype)
    v_out = np.zeros((B, Hkv, out_rows, d), dtype=va.dtype)
    shape = _Shape(B, Hkv, Hkv, d, n_max, 1)
    st = _load().oracle_compact_heads(ctypes.byref(shape), ka.dtype.itemsize, _ptr(ka), _ptr(va), _ptr(idx),
                                      _ptr(kl), out_rows, _ptr(k_out), _ptr(v_out))
    if st != OK:
        raise OracleError("oracle_compact_heads failed with status %d" % st)
    return k_out, v_out


def run_path_layer(q, k, v, lengths, evict_total, pool_kernel, protect, out_rows=None, nthreads=None,
                   kind="dropkv"):
    """S1-S5, the layer-wide selection and the per-head gather."""
    sc = score(q, k, v, lengths, pool_kernel, protect, nthreads=nthreads, kind=kind)
    kept, kl = select_layer(sc["final"], lengths, evict_total, protect)
    rows = int(out_rows) if out_rows is not None else int(kl.max())
    kb, _ = _as_input(k)
    vb, _ = _as_input(v)
    k_out, v_out = compact_heads(kb, vb, kept, kl, rows)
    sc.update(kept_idx=kept, kept_len=kl, k_out=k_out, v_out=v_out)
    return sc


def compact(k, v, kept_idx, kept_len, out_rows: int):
    """Step S7 on raw element bytes.  k, v: numpy arrays [B,Hkv,n_max,d] (any dtype)."""
    ka = np.ascontiguousarray(k)
    va = np.ascontiguousarray(v)
    B, Hkv, n_max, d = ka.shape
    idx = np.ascontiguousarray(kept_idx, dtype=np.int32)
    kl = np.ascontiguousarray(kept_len, dtype=np.int32)
    k_out = np.zeros((B, Hkv, out_rows, d), dtype=ka.dtype)
    v_out = np.zeros((B, Hkv, out_rows, d), dtype=va.dtype)
    shape = _Shape(B, Hkv, Hkv, d, n_max, 1)
    st = _load().oracle_compact(ctypes.byref(shape), ka.dtype.itemsize, _ptr(ka), _ptr(va), _ptr(idx),
                                _ptr(kl), out_rows, _ptr(k_out), _ptr(v_out))
    if st != OK:
        raise OracleError("oracle_compact failed with status %d" % st)
    return k_out, v_out


def run_path(q, k, v, lengths, evict_k, pool_kernel, protect, out_rows=None, nthreads=None, kind="dropkv"):
    """S1-S7 end to end; the kept K/V are gathered from the bf16 inputs."""
    sc = score(q, k, v, lengths, pool_kernel, protect, nthreads=nthreads, kind=kind)
    kept, kl = select(sc["final"], lengths, evict_k, protect)
    rows = int(out_rows) if out_rows is not None else int(kl.max())
    kb, _ = _as_input(k)
    vb, _ = _as_input(v)
    k_out, v_out = compact(kb, vb, kept, kl, rows)
    sc.update(kept_idx=kept, kept_len=kl, k_out=k_out, v_out=v_out)
    return sc
