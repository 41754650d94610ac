"""Thin Python binding of libba.so (ctypes).

Argument marshalling only: tensors are checked for dtype, shape, device and
contiguity and handed to the C ABI as raw pointers together with torch's
current CUDA stream.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback.  If libba.so is missing, importing the
binding raises — call ``build.build()`` (or ``__graft_entry__.build()``)
first.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libba.so")

FAMILY_CODES = {"ttt": 0, "block": 1, "causal": 2}
TABLES = {"token_perm": 0, "anchor_perm": 1, "row_limit": 2, "token_rank": 3,
          "fwd_qtiles": 4, "fwd_segs": 5, "bwd_qtiles": 6, "bwd_kvtiles": 7, "bwd_qranges": 8}
ROLES = {"query": 0, "main_kv": 1, "branch_kv": 2}

STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported", -3: "CUDA error", -4: "device timeout",
    -5: "device bounds", -6: "workspace", -7: "host alloc",
}


class BaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")


class _Desc(ctypes.Structure):
    _fields_ = [
        ("family", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("heads_q", ctypes.c_int32),
        ("heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("cp_degree", ctypes.c_int32),
        ("ttt_depth", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("anchors_per_seq", ctypes.c_int32),
        ("anchors", ctypes.POINTER(ctypes.c_int32)),
    ]


class _Info(ctypes.Structure):
    _fields_ = [
        ("main_tokens", ctypes.c_int64),
        ("branch_queries", ctypes.c_int64),
        ("query_rows", ctypes.c_int64),
        ("main_pairs", ctypes.c_int64),
        ("branch_pairs", ctypes.c_int64),
        ("fwd_flops", ctypes.c_double),
        ("bwd_flops", ctypes.c_double),
        ("fwd_tiles", ctypes.c_int64),
        ("fwd_tile_blocks", ctypes.c_int64),
        ("bwd_kv_tiles", ctypes.c_int64),
        ("comm_bytes_fwd_per_rank", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
    ]


class _KTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


# every symbol the header declares, with its signature
_P = ctypes.c_void_p
_SIGS = {
    "ba_plan_create": (ctypes.c_int, [ctypes.POINTER(_Desc), ctypes.POINTER(_P)]),
    "ba_plan_destroy": (None, [_P]),
    "ba_plan_validate": (ctypes.c_int, [_P]),
    "ba_plan_get_info": (ctypes.c_int, [_P, ctypes.POINTER(_Info)]),
    "ba_plan_get_table": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_int64)]),
    "ba_plan_get_comm_volume": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]),
    "ba_workspace_bytes": (ctypes.c_size_t, [_P]),
    "ba_forward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ba_backward": (ctypes.c_int, [_P] + [_P] * 14 + [ctypes.c_size_t, _P]),
    "ba_workspace_bytes_fp8": (ctypes.c_size_t, [_P]),
    "ba_forward_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ba_forward_step": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "ba_backward_step": (ctypes.c_int, [_P, ctypes.c_int32] + [_P] * 14 + [ctypes.c_size_t, _P]),
    "ba_check_device_status": (ctypes.c_int, [_P, _P, _P]),
    "ba_zigzag_pack": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "ba_lse_merge": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "ba_selftest_wait_timeout": (ctypes.c_int, [_P, _P, ctypes.c_size_t, ctypes.c_int64, _P]),
    "ba_forward_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ba_profile_enable": (ctypes.c_int, [_P, ctypes.c_int32]),
    "ba_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(_KTime), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "ba_last_cuda_error": (ctypes.c_char_p, []),
    "ba_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ba_version": (ctypes.c_char_p, []),
}

_lib = None


def lib():
    """The loaded libba.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libba.so not built ({LIB_PATH}); run branch_attention_speculative_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(rc: int, what: str):
    if rc != 0:
        msg = what
        if rc == -3:
            msg += " [" + lib().ba_last_cuda_error().decode() + "]"
        raise BaError(rc, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _want(t: torch.Tensor, shape, dtype, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: want contiguous cuda {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)} "
                         f"on {t.device} (contiguous={t.is_contiguous()})")


class Plan:
    """A branch-attention problem: zigzag layout, key sets and tile lists."""

    def __init__(self, family: str, cu_seqlens, heads_q: int, heads_kv: int, head_dim: int, cp: int,
                 ttt_depth: int = 0, block_size: int = 0, anchors=None, scale: Optional[float] = None):
        L = lib()
        self.family = family
        self.cu_seqlens = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        self.heads_q, self.heads_kv, self.head_dim, self.cp = heads_q, heads_kv, head_dim, cp
        self.ttt_depth, self.block_size = ttt_depth, block_size
        self.anchors = None if anchors is None else np.ascontiguousarray(np.asarray(anchors, dtype=np.int32))
        self.scale = float(scale if scale is not None else 1.0 / np.sqrt(max(head_dim, 1)))
        S = len(self.cu_seqlens) - 1
        d = _Desc()
        d.family = FAMILY_CODES[family]
        d.num_seqs = S
        d.cu_seqlens = self.cu_seqlens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        d.heads_q, d.heads_kv, d.head_dim = heads_q, heads_kv, head_dim
        d.softmax_scale = self.scale
        d.cp_degree = cp
        d.ttt_depth = ttt_depth
        d.block_size = block_size
        d.anchors_per_seq = 0 if self.anchors is None else len(self.anchors) // max(S, 1)
        d.anchors = (self.anchors.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if self.anchors is not None
                     else ctypes.POINTER(ctypes.c_int32)())
        h = ctypes.c_void_p()
        _check(L.ba_plan_create(ctypes.byref(d), ctypes.byref(h)), "ba_plan_create")
        self._h = h
        self.T = int(self.cu_seqlens[-1])
        self.NA = 0 if self.anchors is None else len(self.anchors)

    @classmethod
    def from_workload(cls, wl) -> "Plan":
        return cls(wl.family, wl.cu_seqlens, wl.heads_q, wl.heads_kv, wl.head_dim, wl.cp,
                   ttt_depth=wl.depth, block_size=wl.block, anchors=wl.anchors, scale=wl.scale)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.ba_plan_destroy(h)
            self._h = None

    # ---- shapes
    def q_shape(self):
        if self.family == "block":
            return (self.NA, self.block_size, self.heads_q, self.head_dim)
        return (self.ttt_depth if self.family == "ttt" else 1, self.T, self.heads_q, self.head_dim)

    def kb_shape(self):
        if self.family == "block":
            return (self.NA, self.block_size, self.heads_kv, self.head_dim)
        if self.family == "ttt":
            return (self.ttt_depth, self.T, self.heads_kv, self.head_dim)
        return None

    def km_shape(self):
        return (self.T, self.heads_kv, self.head_dim)

    # ---- host queries
    def validate(self):
        _check(lib().ba_plan_validate(self._h), "ba_plan_validate")

    def info(self) -> dict:
        inf = _Info()
        _check(lib().ba_plan_get_info(self._h, ctypes.byref(inf)), "ba_plan_get_info")
        return {k: getattr(inf, k) for k, _ in _Info._fields_}

    def table(self, which: str) -> np.ndarray:
        n = ctypes.c_int64()
        _check(lib().ba_plan_get_table(self._h, TABLES[which], None, 0, ctypes.byref(n)), "ba_plan_get_table")
        out = np.zeros(n.value, dtype=np.int32)
        _check(lib().ba_plan_get_table(self._h, TABLES[which], out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       n.value, ctypes.byref(n)), "ba_plan_get_table")
        return out

    def comm_volume(self) -> np.ndarray:
        out = np.zeros(self.cp, dtype=np.int64)
        _check(lib().ba_plan_get_comm_volume(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), self.cp),
               "ba_plan_get_comm_volume")
        return out

    @property
    def workspace_bytes(self) -> int:
        return int(lib().ba_workspace_bytes(self._h))

    def workspace(self, device="cuda") -> torch.Tensor:
        # torch's caching allocator hands out 512-byte aligned blocks
        return torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=device)

    # ---- compute
    def _check_inputs(self, q_b, k_m, v_m, k_b, v_b):
        _want(q_b, self.q_shape(), torch.bfloat16, "q_b")
        _want(k_m, self.km_shape(), torch.bfloat16, "k_m")
        _want(v_m, self.km_shape(), torch.bfloat16, "v_m")
        if self.family != "causal":
            _want(k_b, self.kb_shape(), torch.bfloat16, "k_b")
            _want(v_b, self.kb_shape(), torch.bfloat16, "v_b")

    def forward(self, q_b, k_m, v_m, k_b=None, v_b=None, o=None, lse=None, workspace=None, stream=None):
        """Branch attention forward -> (o bf16 like q_b, lse fp32 q_b.shape[:-1])."""
        self._check_inputs(q_b, k_m, v_m, k_b, v_b)
        if o is None:
            o = torch.empty_like(q_b)
        if lse is None:
            lse = torch.empty(q_b.shape[:-1], dtype=torch.float32, device=q_b.device)
        _want(o, self.q_shape(), torch.bfloat16, "o")
        _want(lse, self.q_shape()[:-1], torch.float32, "lse")
        if workspace is None:
            workspace = self.workspace(q_b.device)
        rc = lib().ba_forward(self._h, _ptr(q_b), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b), _ptr(o), _ptr(lse),
                              _ptr(workspace), workspace.numel(), _stream(stream))
        _check(rc, "ba_forward")
        return o, lse

    @property
    def workspace_bytes_fp8(self) -> int:
        return int(lib().ba_workspace_bytes_fp8(self._h))

    def forward_fp8(self, q_b, k_m, v_m, k_b=None, v_b=None, o=None, lse=None, workspace=None, stream=None):
        """Forward with the main part's QK^T and PV on e4m3 copies (per-tensor
        scales) -> (o bf16, lse fp32); the workspace must hold
        ``workspace_bytes_fp8`` bytes."""
        self._check_inputs(q_b, k_m, v_m, k_b, v_b)
        if o is None:
            o = torch.empty_like(q_b)
        if lse is None:
            lse = torch.empty(q_b.shape[:-1], dtype=torch.float32, device=q_b.device)
        _want(o, self.q_shape(), torch.bfloat16, "o")
        _want(lse, self.q_shape()[:-1], torch.float32, "lse")
        if workspace is None:
            workspace = torch.empty(max(self.workspace_bytes_fp8, 256), dtype=torch.uint8, device=q_b.device)
        rc = lib().ba_forward_fp8(self._h, _ptr(q_b), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b), _ptr(o), _ptr(lse),
                                  _ptr(workspace), workspace.numel(), _stream(stream))
        _check(rc, "ba_forward_fp8")
        return o, lse

    def forward_noalloc(self, q_b, k_m, v_m, k_b=None, v_b=None, o=None, lse=None, stream=None):
        """Forward through ba_forward_noalloc: the library's static scratch array
        replaces the workspace (plans up to 64 MiB of workspace).  Outputs must
        be given or are allocated here, by the caller side, before the call."""
        self._check_inputs(q_b, k_m, v_m, k_b, v_b)
        if o is None:
            o = torch.empty_like(q_b)
        if lse is None:
            lse = torch.empty(q_b.shape[:-1], dtype=torch.float32, device=q_b.device)
        _want(o, self.q_shape(), torch.bfloat16, "o")
        _want(lse, self.q_shape()[:-1], torch.float32, "lse")
        rc = lib().ba_forward_noalloc(self._h, _ptr(q_b), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b), _ptr(o),
                                      _ptr(lse), _stream(stream))
        _check(rc, "ba_forward_noalloc")
        return o, lse

    def backward(self, q_b, k_m, v_m, k_b, v_b, o, lse, d_o, grads=None, workspace=None, stream=None):
        """Branch attention backward -> dict dq_b, dk_m, dv_m, dk_b, dv_b (bf16)."""
        self._check_inputs(q_b, k_m, v_m, k_b, v_b)
        _want(o, self.q_shape(), torch.bfloat16, "o")
        _want(lse, self.q_shape()[:-1], torch.float32, "lse")
        _want(d_o, self.q_shape(), torch.bfloat16, "d_o")
        if grads is None:
            grads = {
                "dq_b": torch.empty_like(q_b),
                "dk_m": torch.empty_like(k_m),
                "dv_m": torch.empty_like(v_m),
                "dk_b": torch.empty_like(k_b) if k_b is not None else None,
                "dv_b": torch.empty_like(v_b) if v_b is not None else None,
            }
        if workspace is None:
            workspace = self.workspace(q_b.device)
        rc = lib().ba_backward(self._h, _ptr(q_b), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b), _ptr(o), _ptr(lse),
                               _ptr(d_o), _ptr(grads["dq_b"]), _ptr(grads["dk_m"]), _ptr(grads["dv_m"]),
                               _ptr(grads.get("dk_b")), _ptr(grads.get("dv_b")), _ptr(workspace),
                               workspace.numel(), _stream(stream))
        _check(rc, "ba_backward")
        return grads

    # ---- EAGLE-3 TTT one step at a time
    def step_shape(self):
        return (self.T, self.heads_q, self.head_dim)

    def forward_step(self, step: int, q_s, k_m, v_m, k_b, v_b, o=None, lse=None, workspace=None, stream=None):
        """TTT step ``step`` alone -> (o_s, lse_s); q_s is that step's [T, Hq, d]
        slice, k_b / v_b the whole [D, T, Hkv, d] buffers (slots > step unread)."""
        if self.family != "ttt":
            raise ValueError("forward_step needs a TTT plan")
        _want(q_s, self.step_shape(), torch.bfloat16, "q_s")
        _want(k_m, self.km_shape(), torch.bfloat16, "k_m")
        _want(v_m, self.km_shape(), torch.bfloat16, "v_m")
        _want(k_b, self.kb_shape(), torch.bfloat16, "k_b")
        _want(v_b, self.kb_shape(), torch.bfloat16, "v_b")
        if o is None:
            o = torch.empty_like(q_s)
        if lse is None:
            lse = torch.empty(q_s.shape[:-1], dtype=torch.float32, device=q_s.device)
        _want(o, self.step_shape(), torch.bfloat16, "o")
        _want(lse, self.step_shape()[:-1], torch.float32, "lse")
        if workspace is None:
            workspace = self.workspace(q_s.device)
        rc = lib().ba_forward_step(self._h, int(step), _ptr(q_s), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b),
                                   _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream))
        _check(rc, "ba_forward_step")
        return o, lse

    def backward_step(self, step: int, q_s, k_m, v_m, k_b, v_b, o_s, lse_s, d_o_s, acc, dq=None, workspace=None,
                      stream=None):
        """Backward of TTT step ``step``: returns dq_s (bf16) and adds the
        step's key gradients into ``acc`` (fp32 dk_m, dv_m, dk_b, dv_b)."""
        if self.family != "ttt":
            raise ValueError("backward_step needs a TTT plan")
        for t, n in ((q_s, "q_s"), (o_s, "o_s"), (d_o_s, "d_o_s")):
            _want(t, self.step_shape(), torch.bfloat16, n)
        _want(lse_s, self.step_shape()[:-1], torch.float32, "lse_s")
        _want(k_m, self.km_shape(), torch.bfloat16, "k_m")
        _want(v_m, self.km_shape(), torch.bfloat16, "v_m")
        _want(k_b, self.kb_shape(), torch.bfloat16, "k_b")
        _want(v_b, self.kb_shape(), torch.bfloat16, "v_b")
        for n, shape in (("dk_m", self.km_shape()), ("dv_m", self.km_shape()), ("dk_b", self.kb_shape()),
                         ("dv_b", self.kb_shape())):
            _want(acc[n], shape, torch.float32, n)
        if dq is None:
            dq = torch.empty_like(q_s)
        if workspace is None:
            workspace = self.workspace(q_s.device)
        rc = lib().ba_backward_step(self._h, int(step), _ptr(q_s), _ptr(k_m), _ptr(v_m), _ptr(k_b), _ptr(v_b),
                                    _ptr(o_s), _ptr(lse_s), _ptr(d_o_s), _ptr(dq), _ptr(acc["dk_m"]),
                                    _ptr(acc["dv_m"]), _ptr(acc["dk_b"]), _ptr(acc["dv_b"]), _ptr(workspace),
                                    workspace.numel(), _stream(stream))
        _check(rc, "ba_backward_step")
        return dq

    def profile(self, enable: bool = True):
        """Turn per-kernel event timing of this plan's launches on or off."""
        _check(lib().ba_profile_enable(self._h, 1 if enable else 0), "ba_profile_enable")

    def profile_read(self) -> dict:
        """{kernel name: (launches, total ms)} since the last read (waits for the events)."""
        buf = (_KTime * 16)()
        n = ctypes.c_int32()
        _check(lib().ba_profile_read(self._h, buf, 16, ctypes.byref(n)), "ba_profile_read")
        return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}

    def selftest_wait_timeout(self, workspace, cycles: int, stream=None):
        """Runs the bounded-wait failure self-test (see include/ba.h)."""
        _check(lib().ba_selftest_wait_timeout(self._h, _ptr(workspace), workspace.numel(), int(cycles),
                                              _stream(stream)), "ba_selftest_wait_timeout")

    def check_device_status(self, workspace, stream=None) -> int:
        return int(lib().ba_check_device_status(self._h, _ptr(workspace), _stream(stream)))

    def zigzag_pack(self, role: str, src, dst=None, inverse=False, workspace=None, stream=None):
        if dst is None:
            dst = torch.empty_like(src)
        if workspace is None:
            workspace = self.workspace(src.device)
        rc = lib().ba_zigzag_pack(self._h, ROLES[role], _ptr(src), _ptr(dst), 1 if inverse else 0, _ptr(workspace),
                                  workspace.numel(), _stream(stream))
        _check(rc, "ba_zigzag_pack")
        return dst


def lse_merge(o_m, l_m, o_b, l_b, stream=None):
    """Eq. 2 on caller tensors: o_* fp32 [rows, d], l_* fp32 [rows] -> (o bf16, l fp32)."""
    rows, d = o_m.shape
    for t, n in ((o_m, "o_m"), (o_b, "o_b")):
        _want(t, (rows, d), torch.float32, n)
    for t, n in ((l_m, "l_m"), (l_b, "l_b")):
        _want(t, (rows,), torch.float32, n)
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=o_m.device)
    l = torch.empty((rows,), dtype=torch.float32, device=o_m.device)
    _check(lib().ba_lse_merge(rows, d, _ptr(o_m), _ptr(l_m), _ptr(o_b), _ptr(l_b), _ptr(o), _ptr(l),
                              _stream(stream)), "ba_lse_merge")
    return o, l


def version() -> str:
    return lib().ba_version().decode()
