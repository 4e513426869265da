"""ctypes binding of libdropkv.so (include/dropkv.h), same names as the C ABI.

Argument marshalling only: tensors are passed as device pointers and the
current torch stream as the CUDA stream; every step runs in the library.  If
the library has not been built, the first call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import _build

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "WORKSPACE", 3: "SINGULAR", 4: "NONFINITE", 5: "CUDA",
                6: "UNSUPPORTED", 7: "DEVICE_ARG", 8: "TIMEOUT"}
FLAG_SINGULAR, FLAG_NONFINITE, FLAG_BAD_LENGTH, FLAG_BAD_K, FLAG_OVERFLOW, FLAG_TIMEOUT = 1, 2, 4, 8, 16, 32


class DropKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s failed: DROPKV_ERR_%s (%d)" % (where, STATUS_NAMES.get(code, "?"), code))
        self.code = code


class dropkv_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n_max", ctypes.c_int32), ("w", ctypes.c_int32)]

    def astuple(self):
        return (self.B, self.Hq, self.Hkv, self.d, self.n_max, self.w)


_lock = threading.Lock()
_lib = None
_active = None          # a library loaded by use_library(), else None


def library_path() -> str:
    return _build.LIB_PATH


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    SH = ctypes.POINTER(dropkv_shape)
    L.dropkv_workspace_size.argtypes = [SH]
    L.dropkv_workspace_size.restype = SZ
    L.dropkv_score.argtypes = [SH, P, P, P, P, I32, I32, P, P, P, SZ, P, P]
    L.dropkv_score.restype = ctypes.c_int
    L.dropkv_score_timed.argtypes = [SH, I32, P, P, P, P, I32, I32, P, P, P, SZ, P, P, P]
    L.dropkv_score_timed.restype = ctypes.c_int
    L.dropkv_score_noalloc.argtypes = [SH, P, P, P, P, I32, I32, P, P, P, P]
    L.dropkv_score_noalloc.restype = ctypes.c_int
    L.dropkv_select.argtypes = [SH, P, P, P, I32, P, P, P, SZ, P, P]
    L.dropkv_select.restype = ctypes.c_int
    L.dropkv_compact.argtypes = [SH, P, P, P, P, I32, P, P, P, P]
    L.dropkv_compact.restype = ctypes.c_int
    L.dropkv_evict.argtypes = [SH, P, P, P, P, P, I32, I32, P, P, P, P, I32, P, P, P, SZ, P, P]
    L.dropkv_evict.restype = ctypes.c_int
    L.dropkv_evict_ex.argtypes = [SH, I32, P, P, P, P, P, I32, I32, P, P, P, P, I32, P, P, P, SZ, P, P]
    L.dropkv_evict_ex.restype = ctypes.c_int
    L.dropkv_evict_prefill.argtypes = [SH, I32, P, P, P, P, P, I32, I32, P, P, P, P, P, I32, P, P, P, SZ, P, P]
    L.dropkv_evict_prefill.restype = ctypes.c_int
    L.dropkv_prefill_attention.argtypes = [SH, P, P, P, P, P, P, SZ, P, P]
    L.dropkv_prefill_attention.restype = ctypes.c_int
    L.dropkv_score_ex.argtypes = [SH, I32, P, P, P, P, I32, I32, P, P, P, SZ, P, P]
    L.dropkv_score_ex.restype = ctypes.c_int
    L.dropkv_select_layer.argtypes = [SH, P, P, P, I32, P, P, P, SZ, P, P]
    L.dropkv_select_layer.restype = ctypes.c_int
    L.dropkv_compact_heads.argtypes = [SH, P, P, P, P, I32, P, P, P, P]
    L.dropkv_compact_heads.restype = ctypes.c_int
    L.dropkv_read_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    L.dropkv_read_status.restype = ctypes.c_int
    L.dropkv_version.argtypes = []
    L.dropkv_version.restype = ctypes.c_char_p
    for hook in ("dropkv_test_skip_pass2_k", "dropkv_test_skip_prefill_k"):
        if hasattr(L, hook):
            getattr(L, hook).argtypes = [I32, I32]
            getattr(L, hook).restype = ctypes.c_int
    return L


def lib():
    """The library the calls go to: libdropkv.so (raises if it was not
    built), or the one a use_library() block selected."""
    global _lib
    if _active is not None:
        return _active
    with _lock:
        if _lib is None:
            _lib = _load(_build.LIB_PATH)
    return _lib


class use_library:
    """Route this module's calls to another build of the library (the test
    build of include/dropkv_test_hooks.h) inside a with-block."""

    _cache = {}

    def __init__(self, path):
        with _lock:
            if path not in self._cache:
                self._cache[path] = _load(path)
        self.L = self._cache[path]

    def __enter__(self):
        global _active
        self.prev, _active = _active, self.L
        return self.L

    def __exit__(self, *exc):
        global _active
        _active = self.prev
        return False


def declared_functions(header: str = None):
    """Names of the functions include/dropkv.h declares."""
    header = header or os.path.join(_build.INCLUDE, "dropkv.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dropkv_[a-z0-9_]+)\s*\(", text)))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_shape(B, Hq, Hkv, d, n_max, w) -> dropkv_shape:
    return dropkv_shape(int(B), int(Hq), int(Hkv), int(d), int(n_max), int(w))


def _check(code, where):
    if code != 0:
        raise DropKVError(code, where)
    return code


def dropkv_workspace_size(shape: dropkv_shape) -> int:
    return int(lib().dropkv_workspace_size(ctypes.byref(shape)))


def dropkv_score(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace, status,
                 stream=None):
    code = lib().dropkv_score(ctypes.byref(shape), _ptr(q_window), _ptr(k), _ptr(v), _ptr(lengths),
                              int(pool_kernel), int(protect), _ptr(scores), _ptr(raw_scores), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    return _check(code, "dropkv_score")


def dropkv_score_timed(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                       status, events, stream=None, kind="dropkv"):
    """dropkv_score recording 5 torch.cuda.Event objects at its phase boundaries."""
    if len(events) != 5:
        raise ValueError("dropkv_score_timed records 5 events")
    arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    code = lib().dropkv_score_timed(ctypes.byref(shape), SCORE_KINDS[kind], _ptr(q_window), _ptr(k), _ptr(v),
                                    _ptr(lengths),
                                    int(pool_kernel), int(protect), _ptr(scores), _ptr(raw_scores),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                                    _stream(stream), arr)
    return _check(code, "dropkv_score_timed")


def dropkv_score_noalloc(shape, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, status,
                         stream=None):
    """dropkv_score with the library's fixed scratch array instead of a workspace (allocates nothing)."""
    code = lib().dropkv_score_noalloc(ctypes.byref(shape), _ptr(q_window), _ptr(k), _ptr(v), _ptr(lengths),
                                      int(pool_kernel), int(protect), _ptr(scores), _ptr(raw_scores),
                                      _ptr(status), _stream(stream))
    return _check(code, "dropkv_score_noalloc")


def dropkv_select(shape, scores, lengths, evict_k, protect, kept_idx, kept_len, workspace, status, stream=None):
    code = lib().dropkv_select(ctypes.byref(shape), _ptr(scores), _ptr(lengths), _ptr(evict_k), int(protect),
                               _ptr(kept_idx), _ptr(kept_len), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    return _check(code, "dropkv_select")


def dropkv_compact(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream=None):
    code = lib().dropkv_compact(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(kept_idx), _ptr(kept_len),
                                int(out_rows), _ptr(k_out), _ptr(v_out), _ptr(status), _stream(stream))
    return _check(code, "dropkv_compact")


def dropkv_evict(shape, q_window, k, v, lengths, evict_k, pool_kernel, protect, scores, raw_scores, kept_idx,
                 kept_len, out_rows, k_out, v_out, workspace, status, stream=None):
    code = lib().dropkv_evict(ctypes.byref(shape), _ptr(q_window), _ptr(k), _ptr(v), _ptr(lengths), _ptr(evict_k),
                              int(pool_kernel), int(protect), _ptr(scores), _ptr(raw_scores), _ptr(kept_idx),
                              _ptr(kept_len), int(out_rows), _ptr(k_out), _ptr(v_out), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    return _check(code, "dropkv_evict")


SCORE_KINDS = {"dropkv": 0, "snapkv": 1}


def dropkv_score_ex(shape, kind, q_window, k, v, lengths, pool_kernel, protect, scores, raw_scores, workspace,
                    status, stream=None):
    code = lib().dropkv_score_ex(ctypes.byref(shape), SCORE_KINDS[kind], _ptr(q_window), _ptr(k), _ptr(v),
                                 _ptr(lengths), int(pool_kernel), int(protect), _ptr(scores), _ptr(raw_scores),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                                 _stream(stream))
    return _check(code, "dropkv_score_ex")


def dropkv_evict_ex(shape, kind, q_window, k, v, lengths, evict_k, pool_kernel, protect, scores, raw_scores,
                    kept_idx, kept_len, out_rows, k_out, v_out, workspace, status, stream=None):
    code = lib().dropkv_evict_ex(ctypes.byref(shape), SCORE_KINDS[kind], _ptr(q_window), _ptr(k), _ptr(v),
                                 _ptr(lengths), _ptr(evict_k), int(pool_kernel), int(protect), _ptr(scores),
                                 _ptr(raw_scores), _ptr(kept_idx), _ptr(kept_len), int(out_rows), _ptr(k_out),
                                 _ptr(v_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(status), _stream(stream))
    return _check(code, "dropkv_evict_ex")


def dropkv_evict_prefill(shape, kind, q, k, v, lengths, evict_k, pool_kernel, protect, attn_out, scores, raw_scores,
                         kept_idx, kept_len, out_rows, k_out, v_out, workspace, status, stream=None):
    _check(lib().dropkv_evict_prefill(ctypes.byref(shape), SCORE_KINDS[kind], _ptr(q), _ptr(k), _ptr(v), _ptr(lengths),
                                      _ptr(evict_k), int(pool_kernel), int(protect), _ptr(attn_out), _ptr(scores),
                                      _ptr(raw_scores), _ptr(kept_idx), _ptr(kept_len), int(out_rows), _ptr(k_out),
                                      _ptr(v_out), _ptr(workspace), workspace.numel(), _ptr(status),
                                      _stream(stream)), "dropkv_evict_prefill")


def dropkv_prefill_attention(shape, q, k, v, lengths, attn_out, workspace, status, stream=None):
    _check(lib().dropkv_prefill_attention(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(lengths),
                                          _ptr(attn_out), _ptr(workspace), workspace.numel(), _ptr(status),
                                          _stream(stream)), "dropkv_prefill_attention")


def dropkv_select_layer(shape, scores, lengths, evict_total, protect, kept_idx, kept_len, workspace, status,
                        stream=None):
    code = lib().dropkv_select_layer(ctypes.byref(shape), _ptr(scores), _ptr(lengths), _ptr(evict_total),
                                     int(protect), _ptr(kept_idx), _ptr(kept_len), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    return _check(code, "dropkv_select_layer")


def dropkv_compact_heads(shape, k, v, kept_idx, kept_len, out_rows, k_out, v_out, status, stream=None):
    code = lib().dropkv_compact_heads(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(kept_idx), _ptr(kept_len),
                                      int(out_rows), _ptr(k_out), _ptr(v_out), _ptr(status), _stream(stream))
    return _check(code, "dropkv_compact_heads")


def dropkv_read_status(status, stream=None):
    """Sync the stream and return (status code, raw flag word)."""
    flags = ctypes.c_uint32(0)
    code = lib().dropkv_read_status(_ptr(status), _stream(stream), ctypes.byref(flags))
    return int(code), int(flags.value)


def dropkv_version() -> str:
    return lib().dropkv_version().decode()
