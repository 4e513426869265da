"""User-facing wrapper: allocate with torch, run score -> select -> compact.

Every computation runs in libdropkv.so; this module only owns buffers.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding as B


class DropKV:
    """Reusable buffers for one problem shape on one device.

    run() takes device tensors q_window [B,Hq,w,d], k, v [B,Hkv,n_max,d] (bf16),
    lengths [B] int32 (or None) and evict_k [B] int32, and returns the final
    scores, kept indices and lengths and the compacted K/V."""

    def __init__(self, B_: int, Hq: int, Hkv: int, d: int, n_max: int, w: int, pool_kernel: int = 5,
                 protect: Optional[int] = None, out_rows: Optional[int] = None, device=None, kind: str = "dropkv"):
        """kind: "dropkv" (the perturbation score) or "snapkv" (window sum of
        attention probabilities, the attention-only baseline)."""
        if kind not in B.SCORE_KINDS:
            raise ValueError("kind must be one of %s" % sorted(B.SCORE_KINDS))
        self.kind = kind
        self.shape = B.make_shape(B_, Hq, Hkv, d, n_max, w)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.pool_kernel = int(pool_kernel)
        self.protect = int(w if protect is None else protect)
        self.out_rows = int(n_max if out_rows is None else out_rows)
        with torch.cuda.device(self.device):
            ws = B.dropkv_workspace_size(self.shape)
            if ws == 0:
                raise B.DropKVError(6, "dropkv_workspace_size")
            dev = self.device
            self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
            self.status = torch.zeros(1, dtype=torch.int32, device=dev)
            self.scores = torch.empty(B_, Hkv, n_max, dtype=torch.float32, device=dev)
            self.raw_scores = torch.empty(B_, Hkv, n_max, dtype=torch.float32, device=dev)
            self.kept_idx = torch.empty(B_, Hkv, n_max, dtype=torch.int32, device=dev)
            self.kept_len = torch.empty(B_, dtype=torch.int32, device=dev)
            self.kept_len_heads = torch.empty(B_, Hkv, dtype=torch.int32, device=dev)
            self.k_out = torch.empty(B_, Hkv, self.out_rows, d, dtype=torch.bfloat16, device=dev)
            self.v_out = torch.empty(B_, Hkv, self.out_rows, d, dtype=torch.bfloat16, device=dev)

    def window_stats(self):
        """(lse [B,Hkv,R], a [B,Hkv,R,d]) from the last score() call (views of the workspace)."""
        Bn, Hq, Hkv, d, _, w = self.shape.astuple()
        R = (Hq // Hkv) * w
        U = Bn * Hkv
        lse = self.workspace[: U * R * 4].view(torch.float32).view(Bn, Hkv, R)
        off = (U * R * 4 + 255) // 256 * 256
        a = self.workspace[off: off + U * R * d * 4].view(torch.float32).view(Bn, Hkv, R, d)
        return lse, a

    def score(self, q, k, v, lengths=None, stream=None, keep_raw=True):
        B.dropkv_score_ex(self.shape, self.kind, q, k, v, lengths, self.pool_kernel, self.protect, self.scores,
                          self.raw_scores if keep_raw else None, self.workspace, self.status, stream)

    def select(self, lengths, evict_k, stream=None):
        B.dropkv_select(self.shape, self.scores, lengths, evict_k, self.protect, self.kept_idx, self.kept_len,
                        self.workspace, self.status, stream)

    def compact(self, k, v, stream=None):
        B.dropkv_compact(self.shape, k, v, self.kept_idx, self.kept_len, self.out_rows, self.k_out, self.v_out,
                         self.status, stream)

    def run(self, q, k, v, lengths, evict_k, stream=None, keep_raw=True):
        """The whole step in one library call (dropkv_evict)."""
        B.dropkv_evict_ex(self.shape, self.kind, q, k, v, lengths, evict_k, self.pool_kernel, self.protect,
                          self.scores, self.raw_scores if keep_raw else None, self.kept_idx, self.kept_len,
                          self.out_rows, self.k_out, self.v_out, self.workspace, self.status, stream)

    def run_prefill(self, q, k, v, lengths, evict_k, attn_out, stream=None, keep_raw=True):
        """The prompt's causal attention over every query row q [B,Hq,n_max,d]
        (output into attn_out, same shape and dtype) with the eviction fused in:
        the window statistics come from its last w rows (dropkv_evict_prefill)."""
        B.dropkv_evict_prefill(self.shape, self.kind, q, k, v, lengths, evict_k, self.pool_kernel, self.protect,
                               attn_out, self.scores, self.raw_scores if keep_raw else None, self.kept_idx,
                               self.kept_len, self.out_rows, self.k_out, self.v_out, self.workspace, self.status,
                               stream)

    def prefill_attention(self, q, k, v, lengths, attn_out, stream=None):
        """The prompt's causal attention alone (dropkv_prefill_attention)."""
        B.dropkv_prefill_attention(self.shape, q, k, v, lengths, attn_out, self.workspace, self.status, stream)

    def run_separate(self, q, k, v, lengths, evict_k, stream=None, keep_raw=True):
        """The same step as three library calls (score, select, compact)."""
        self.score(q, k, v, lengths, stream, keep_raw)
        self.select(lengths, evict_k, stream)
        self.compact(k, v, stream)

    def select_layer(self, lengths, evict_total, stream=None):
        """Layer-wide selection (one pool per sequence over its KV heads):
        kept_idx per head, counts in kept_len_heads [B, Hkv]."""
        B.dropkv_select_layer(self.shape, self.scores, lengths, evict_total, self.protect, self.kept_idx,
                              self.kept_len_heads, self.workspace, self.status, stream)

    def compact_heads(self, k, v, stream=None):
        B.dropkv_compact_heads(self.shape, k, v, self.kept_idx, self.kept_len_heads, self.out_rows, self.k_out,
                               self.v_out, self.status, stream)

    def run_layer(self, q, k, v, lengths, evict_total, stream=None, keep_raw=True):
        """Score, layer-wide selection and per-head compaction (AdaDropKV reading)."""
        self.score(q, k, v, lengths, stream, keep_raw)
        self.select_layer(lengths, evict_total, stream)
        self.compact_heads(k, v, stream)

    def check(self, stream=None):
        """Sync and raise if the device status word reports an error."""
        code, flags = B.dropkv_read_status(self.status, stream)
        if code != 0:
            raise B.DropKVError(code, "device status 0x%x" % flags)
        return flags

    def reset_status(self):
        self.status.zero_()
