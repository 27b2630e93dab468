"""ctypes binding of libanchorattn.so: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; torch supplies the
device memory and the stream. There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libanchorattn.so")

MASK_CAUSAL, MASK_INTRA_DOC, MASK_ANCHOR = 0, 1, 2
POS_RESET, POS_CONTINUOUS = 0, 1
ROPE_ADJACENT, ROPE_HALF, ROPE_NONE = 0, 1, 2
STATUS = {0: "AA_OK", 1: "AA_ERR_INVALID_ARG", 2: "AA_ERR_UNSUPPORTED", 3: "AA_ERR_CUDA",
          4: "AA_ERR_NO_MEMORY", 5: "AA_ERR_TIMEOUT"}

# every symbol include/anchorattn.h declares
EXPORTS = ["aa_plan", "aa_plan_with_theta", "aa_plan_segments", "aa_plan_destroy", "aa_plan_metadata", "aa_plan_stats", "aa_plan_work",
           "aa_rope_apply", "aa_fwd", "aa_fwd_workspace_bytes", "aa_bwd_workspace_bytes", "aa_bwd", "aa_bwd_from_fwd",
           "aa_bwd_from_fwd_workspace_bytes", "aa_bwd_static_workspace", "aa_check_device_error",
           "aa_set_wait_limit", "aa_set_bwd_timing_events", "aa_selftest_bounded_wait", "aa_status_string",
           "aa_last_error", "aa_shift_diag_workspace_bytes", "aa_shift_diag", "aa_shard_plan"]


class AAShardPiece(ctypes.Structure):
    _fields_ = [("shard", ctypes.c_int32), ("doc", ctypes.c_int32), ("kv_head_begin", ctypes.c_int32),
                ("kv_head_end", ctypes.c_int32), ("cost", ctypes.c_int64)]


class AAConfig(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("softmax_scale", ctypes.c_float),
                ("pos_shift", ctypes.c_int32), ("mask_mode", ctypes.c_int32),
                ("pos_mode", ctypes.c_int32), ("rope_layout", ctypes.c_int32),
                ("host_only", ctypes.c_int32)]


class AAError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib():
    """Load libanchorattn.so (built by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)
        i32p = ctypes.POINTER(ctypes.c_int32)
        sig = {
            "aa_plan": ([ctypes.POINTER(AAConfig), i32p, i32, vp, ctypes.POINTER(vp)], ctypes.c_int),
            "aa_plan_with_theta": ([ctypes.POINTER(AAConfig), i32p, i32, ctypes.POINTER(ctypes.c_double), vp,
                                    ctypes.POINTER(vp)], ctypes.c_int),
            "aa_plan_segments": ([ctypes.POINTER(AAConfig), i32p, vp, ctypes.POINTER(vp)], ctypes.c_int),
            "aa_plan_destroy": ([vp], ctypes.c_int),
            "aa_plan_metadata": ([vp, i32p, i32p], ctypes.c_int),
            "aa_plan_stats": ([vp, i64p, i64p, i64p], ctypes.c_int),
            "aa_plan_work": ([vp, i64p, i64p], ctypes.c_int),
            "aa_rope_apply": ([vp, vp, vp, i32, i32, vp], ctypes.c_int),
            "aa_fwd": ([vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
            "aa_fwd_workspace_bytes": ([vp], ctypes.c_size_t),
            "aa_bwd_workspace_bytes": ([vp], ctypes.c_size_t),
            "aa_bwd": ([vp] + [vp] * 9 + [vp, ctypes.c_size_t, vp], ctypes.c_int),
            "aa_bwd_from_fwd": ([vp] + [vp] * 8 + [vp, ctypes.c_size_t, vp], ctypes.c_int),
            "aa_bwd_from_fwd_workspace_bytes": ([vp], ctypes.c_size_t),
            "aa_bwd_static_workspace": ([vp] + [vp] * 9 + [vp], ctypes.c_int),
            "aa_check_device_error": ([vp, vp], ctypes.c_int),
            "aa_set_wait_limit": ([vp, ctypes.c_uint64], ctypes.c_int),
            "aa_set_bwd_timing_events": ([vp, vp, vp], ctypes.c_int),
            "aa_selftest_bounded_wait": ([vp, vp], ctypes.c_int),
            "aa_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "aa_last_error": ([], ctypes.c_char_p),
            "aa_shift_diag_workspace_bytes": ([vp], ctypes.c_size_t),
            "aa_shift_diag": ([vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
            "aa_shard_plan": ([i32p, i32, i32, i32, i32, ctypes.POINTER(AAShardPiece), i32, i32p, i64p],
                              ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


def _check(status):
    if status != 0:
        raise AAError(status, lib().aa_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """aa_plan for one packing; compute methods wrap aa_rope_apply/aa_fwd/aa_bwd."""

    def __init__(self, cu_doclens, total_tokens, num_q_heads, num_kv_heads, head_dim,
                 rope_base=1e4, mask_mode=MASK_ANCHOR, pos_mode=POS_RESET,
                 rope_layout=ROPE_ADJACENT, softmax_scale=0.0, pos_shift=0,
                 host_only=False, stream=None, theta=None, doc_of_token=None):
        """theta: optional [head_dim / 2] rotation frequencies (aa_plan_with_theta)
        replacing rope_base^(-2p/D), e.g. an NTK- or YaRN-scaled table.
        doc_of_token: optional int32 [T] document id per token (aa_plan_segments;
        token 0 = 0, the anchor); cu_doclens is then ignored."""
        self.cfg = AAConfig(int(total_tokens), int(num_q_heads), int(num_kv_heads), int(head_dim),
                            float(rope_base), float(softmax_scale or 0.0), int(pos_shift),
                            int(mask_mode), int(pos_mode), int(rope_layout), int(bool(host_only)))
        self.T, self.Hq, self.Hkv, self.D = int(total_tokens), int(num_q_heads), int(num_kv_heads), int(head_dim)
        self.host_only = bool(host_only)
        if cu_doclens is None:
            cu, n = None, 0
        else:
            self._cu = np.ascontiguousarray(np.asarray(cu_doclens, dtype=np.int32))
            cu = self._cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            n = int(self._cu.size) - 1
        h = ctypes.c_void_p()
        st = ctypes.c_void_p(0) if host_only else _stream(stream)
        if doc_of_token is not None:
            if theta is not None:
                raise ValueError("doc_of_token and theta cannot be combined")
            self._doc = np.ascontiguousarray(np.asarray(doc_of_token, dtype=np.int32))
            if self._doc.shape != (self.T,):
                raise ValueError("doc_of_token must have total_tokens entries")
            _check(lib().aa_plan_segments(ctypes.byref(self.cfg),
                                          self._doc.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), st,
                                          ctypes.byref(h)))
        elif theta is None:
            _check(lib().aa_plan(ctypes.byref(self.cfg), cu, n, st, ctypes.byref(h)))
        else:
            self._theta = np.ascontiguousarray(np.asarray(theta, dtype=np.float64))
            if self._theta.shape != (self.D // 2,):
                raise ValueError(f"theta must have head_dim / 2 = {self.D // 2} entries")
            _check(lib().aa_plan_with_theta(ctypes.byref(self.cfg), cu, n,
                                            self._theta.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), st,
                                            ctypes.byref(h)))
        self._h = h

    # ---- lifetime
    def close(self):
        if getattr(self, "_h", None):
            lib().aa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---- host queries
    def metadata(self):
        doc = np.zeros(self.T, dtype=np.int32)
        pos = np.zeros(self.T, dtype=np.int32)
        _check(lib().aa_plan_metadata(self._h, doc.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                      pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return doc, pos

    def stats(self):
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().aa_plan_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
        return {"unmasked_pairs": a.value, "live_tiles": b.value, "causal_tiles": c.value}

    def work(self):
        a, b = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().aa_plan_work(self._h, ctypes.byref(a), ctypes.byref(b)))
        return {"fwd_tiles": a.value, "bwd_tiles": b.value}

    def workspace_bytes(self):
        return int(lib().aa_bwd_workspace_bytes(self._h))

    def set_wait_limit(self, ns):
        _check(lib().aa_set_wait_limit(self._h, int(ns)))

    def set_bwd_timing_events(self, start=None, stop=None):
        """torch.cuda.Event pair (enable_timing=True) recorded around the main bwd kernel."""
        if start is not None and (not start.cuda_event or not stop.cuda_event):
            raise ValueError("record the events once with torch first so that they exist")
        a = ctypes.c_void_p(start.cuda_event) if start is not None else None
        b = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
        _check(lib().aa_set_bwd_timing_events(self._h, a, b))

    def selftest_bounded_wait(self, stream=None):
        _check(lib().aa_selftest_bounded_wait(self._h, _stream(stream)))

    def check_device_error(self, stream=None):
        _check(lib().aa_check_device_error(self._h, _stream(stream)))

    # ---- compute (device tensors only)
    def rope_apply(self, x, inverse=False, out=None, stream=None):
        import torch
        assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
        y = torch.empty_like(x) if out is None else out
        _check(lib().aa_rope_apply(self._h, _ptr(x), _ptr(y), int(x.shape[1]), int(bool(inverse)),
                                   _stream(stream)))
        return y

    def fwd_workspace_bytes(self):
        return int(lib().aa_fwd_workspace_bytes(self._h))

    def alloc_fwd_workspace(self, device):
        import torch
        return torch.empty(max(self.fwd_workspace_bytes(), 256), device=device, dtype=torch.uint8)

    def fwd(self, q, k, v, o=None, lse=None, workspace=None, stream=None):
        import torch
        for t in (q, k, v):
            assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
        o = torch.empty_like(q) if o is None else o
        lse = torch.empty(self.Hq, self.T, device=q.device, dtype=torch.float32) if lse is None else lse
        ws = self.alloc_fwd_workspace(q.device) if workspace is None else workspace
        _check(lib().aa_fwd(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws),
                            ctypes.c_size_t(ws.numel()), _stream(stream)))
        return o, lse

    def alloc_workspace(self, device):
        import torch
        return torch.empty(self.workspace_bytes(), device=device, dtype=torch.uint8)

    def bwd(self, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, workspace=None, stream=None):
        import torch
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        ws = self.alloc_workspace(q.device) if workspace is None else workspace
        _check(lib().aa_bwd(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ctypes.c_size_t(ws.numel()),
                            _stream(stream)))
        return dq, dk, dv

    def bwd_from_fwd_workspace_bytes(self):
        return int(lib().aa_bwd_from_fwd_workspace_bytes(self._h))

    def bwd_from_fwd(self, fwd_workspace, v, o, lse, dout, dq=None, dk=None, dv=None, workspace=None,
                     stream=None):
        """aa_bwd_from_fwd: the backward pass reading the rotated Q and K that
        aa_fwd left in ``fwd_workspace`` (the tensor passed to fwd(); q and k
        are not needed). Same results as bwd()."""
        import torch
        dq = torch.empty_like(o) if dq is None else dq
        dk = torch.empty_like(v) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        if workspace is None:
            workspace = torch.empty(max(self.bwd_from_fwd_workspace_bytes(), 256), device=v.device,
                                    dtype=torch.uint8)
        _check(lib().aa_bwd_from_fwd(self._h, _ptr(fwd_workspace), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                     ctypes.c_size_t(workspace.numel()), _stream(stream)))
        return dq, dk, dv

    def shift_diag(self, other, q, k, workspace=None, stream=None):
        """aa_shift_diag: Eq. 4 / Eq. 5 shift discrepancies between this plan's
        pos_shift and ``other``'s (same problem otherwise) for un-rotated q, k.
        Returns (col [Hq, T], first [Hq, T], result) with result = float64
        [D, D_logit, D_0, L_0, D_1, L_1, ...] on the device."""
        import torch
        for t in (q, k):
            assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
        col = torch.empty(self.Hq, self.T, device=q.device, dtype=torch.float32)
        first = torch.empty_like(col)
        res = torch.empty(2 + 2 * self.Hq, device=q.device, dtype=torch.float64)
        need = int(lib().aa_shift_diag_workspace_bytes(self._h))
        ws = torch.empty(max(need, 256), device=q.device, dtype=torch.uint8) if workspace is None else workspace
        _check(lib().aa_shift_diag(self._h, other._h, _ptr(q), _ptr(k), _ptr(col), _ptr(first), _ptr(res),
                                   _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream)))
        return col, first, res

    def bwd_static_workspace(self, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, stream=None):
        """aa_bwd_static_workspace: the backward pass with the library's static
        64 MiB scratch instead of a caller-provided workspace (for callers that
        must not allocate device memory; outputs may still come from torch)."""
        import torch
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        _check(lib().aa_bwd_static_workspace(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
        return dq, dk, dv


def shard_plan(cu_doclens, num_kv_heads, group, num_shards):
    """aa_shard_plan: pieces (shard, doc, kv_head_begin, kv_head_end, cost) and
    each shard's total cost. Host only."""
    cu = np.ascontiguousarray(np.asarray(cu_doclens, dtype=np.int32))
    n = ctypes.c_int32()
    ip = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    st = lib().aa_shard_plan(ip(cu), int(cu.size) - 1, int(num_kv_heads), int(group), int(num_shards), None, 0,
                             ctypes.byref(n), None)
    if st != 0 and n.value == 0:
        _check(st)
    pieces = (AAShardPiece * max(n.value, 1))()
    cost = np.zeros(int(num_shards), dtype=np.int64)
    _check(lib().aa_shard_plan(ip(cu), int(cu.size) - 1, int(num_kv_heads), int(group), int(num_shards), pieces,
                               n.value, ctypes.byref(n), cost.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
    out = [(p.shard, p.doc, p.kv_head_begin, p.kv_head_end, p.cost) for p in pieces[:n.value]]
    return out, cost
