"""Python binding of liblora_sgmv.so (GB300 / sm_103a SGMV LoRA).

Argument marshalling only: every step of the computation runs in the CUDA
library; this module turns torch tensors into pointers, strides and the
current CUDA stream, calls the C ABI declared in ``include/lora_sgmv.h`` and
raises ``LoraError`` on any non-OK status.  There is no fallback: if the
library cannot be loaded, every call raises.

Names follow the C ABI: ``lora_build_routing``, ``lora_set_slot``,
``lora_shrink``, ``lora_expand``, ``lora_workspace_bytes``,
``lora_sgmv_apply``, ``lora_sgmv_apply_noalloc``, ``lora_base_gemm_apply``,
``lora_get_device_status``, ``lora_last_call_path``, ``lora_status_string``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblora_sgmv.so")

LORA_OK = 0
STATUS_NAMES = {0: "LORA_OK", 1: "LORA_ERR_NULL", 2: "LORA_ERR_SHAPE", 3: "LORA_ERR_RANK",
                4: "LORA_ERR_SLOT_RANGE", 5: "LORA_ERR_ROUTING", 6: "LORA_ERR_DTYPE",
                7: "LORA_ERR_ALIGN", 8: "LORA_ERR_WORKSPACE", 9: "LORA_ERR_CUDA",
                10: "LORA_ERR_TOO_MANY_GROUPS"}
DTYPE_F32, DTYPE_BF16 = 0, 1
DEV_BAD_SLOT, DEV_BAD_OFFSETS, DEV_BAD_END, DEV_TIMEOUT, DEV_BAD_ROW = 1, 2, 4, 8, 16
# Kernel families of lora_last_call_path (include/lora_sgmv.h).
PATH_GENERIC_SHRINK, PATH_GENERIC_EXPAND = 0x1, 0x2
PATH_MMA_SHRINK, PATH_MMA_EXPAND = 0x4, 0x8
PATH_TC_SHRINK, PATH_TC_EXPAND = 0x10, 0x20
PATH_PREP, PATH_BASE_GEMM = 0x80, 0x100
MAX_SLICES = 3


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, STATUS_NAMES.get(status, str(status))))


class _Slice(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("A_slot_stride", ctypes.c_int64), ("B", ctypes.c_void_p),
                ("B_slot_stride", ctypes.c_int64), ("out_dim", ctypes.c_int32), ("y", ctypes.c_void_p),
                ("y_row_stride", ctypes.c_int64), ("bias", ctypes.c_void_p), ("bias_slot_stride", ctypes.c_int64)]


class _Problem(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("num_tokens", ctypes.c_int32), ("in_dim", ctypes.c_int32),
                ("max_num_loras", ctypes.c_int32), ("max_lora_rank", ctypes.c_int32),
                ("x", ctypes.c_void_p), ("x_row_stride", ctypes.c_int64),
                ("num_slices", ctypes.c_int32), ("slices", _Slice * MAX_SLICES), ("slot_ranks", ctypes.c_void_p)]


class _BaseWeight(ctypes.Structure):
    _fields_ = [("W0", ctypes.c_void_p), ("row_stride", ctypes.c_int64)]


class _Routing(ctypes.Structure):
    _fields_ = [("lora_ids", ctypes.c_void_p), ("grouped_offsets", ctypes.c_void_p),
                ("num_groups", ctypes.c_int32), ("end", ctypes.c_int32), ("token_rows", ctypes.c_void_p),
                ("host_grouped_offsets", ctypes.c_void_p), ("host_lora_ids", ctypes.c_void_p)]


_lib = None
_load_error = None


def library_path() -> str:
    return LIB_PATH


def lib():
    """The loaded library; raises if it is missing or fails to load."""
    global _lib, _load_error
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("liblora_sgmv.so is not built (run adapter_sgmv_lora_gb300/build.py or "
                           "__graft_entry__.build()); there is no fallback")
    L = ctypes.CDLL(LIB_PATH)
    i32 = ctypes.c_int32
    i32p = ctypes.POINTER(ctypes.c_int32)
    vp = ctypes.c_void_p
    L.lora_build_routing.restype = ctypes.c_int
    L.lora_build_routing.argtypes = [i32, i32p, i32p, i32, i32p, i32p, i32p, i32p, i32p, i32p]
    L.lora_build_token_rows.restype = ctypes.c_int
    L.lora_build_token_rows.argtypes = [i32, i32p, i32p, i32, i32p]
    L.lora_set_slot_bias.restype = ctypes.c_int
    L.lora_set_slot_bias.argtypes = [ctypes.POINTER(_Problem), i32, i32, vp, ctypes.c_int, vp]
    L.lora_set_slot.restype = ctypes.c_int
    L.lora_set_slot.argtypes = [ctypes.POINTER(_Problem), i32, i32, i32, ctypes.c_double, i32, vp, vp,
                                ctypes.c_int, vp]
    for name in ("lora_shrink", "lora_expand"):
        f = getattr(L, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(_Routing), vp, vp]
    L.lora_workspace_bytes.restype = ctypes.c_size_t
    L.lora_workspace_bytes.argtypes = [ctypes.POINTER(_Problem), i32]
    L.lora_sgmv_apply.restype = ctypes.c_int
    L.lora_sgmv_apply.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(_Routing), vp,
                                  ctypes.c_size_t, vp]
    L.lora_sgmv_apply_noalloc.restype = ctypes.c_int
    L.lora_sgmv_apply_noalloc.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(_Routing), vp]
    L.lora_get_device_status.restype = ctypes.c_int
    L.lora_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.lora_status_string.restype = ctypes.c_char_p
    L.lora_status_string.argtypes = [ctypes.c_int]
    L.lora_base_gemm_apply.restype = ctypes.c_int
    L.lora_base_gemm_apply.argtypes = [ctypes.POINTER(_Problem), ctypes.POINTER(_Routing),
                                       ctypes.POINTER(_BaseWeight), vp, ctypes.c_size_t, vp]
    L.lora_last_call_path.restype = ctypes.c_uint32
    L.lora_last_call_path.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.lora_selftest_wait_timeout.restype = ctypes.c_int
    L.lora_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != LORA_OK:
        raise LoraError(rc, what)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


# --------------------------------------------------------------- routing --

def lora_build_routing(req_slot, req_num_tokens, max_num_loras: int, out_ids=None, out_offsets=None) -> dict:
    """Host sort + group (see include/lora_sgmv.h).  Returns numpy arrays.

    out_ids / out_offsets (optional): contiguous int32 arrays of at least
    max_num_loras and max_num_loras + 1 elements (for instance views of
    pinned host tensors) that receive lora_ids and grouped_offsets directly;
    the returned entries are then views of them."""
    L = lib()
    slots = np.ascontiguousarray(np.asarray(req_slot, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(req_num_tokens, dtype=np.int32))
    if slots.shape != lens.shape or slots.ndim != 1:
        raise ValueError("req_slot and req_num_tokens must be 1-D and the same length")
    n = int(slots.size)
    S = int(max_num_loras)
    perm = np.zeros(max(n, 1), dtype=np.int32)
    for a, need, name in ((out_ids, max(S, 1), "out_ids"), (out_offsets, max(S, 1) + 1, "out_offsets")):
        if a is not None and (a.dtype != np.int32 or a.ndim != 1 or a.size < need or not a.flags.c_contiguous):
            raise ValueError("%s must be a contiguous int32 array of at least %d elements" % (name, need))
    ids = out_ids if out_ids is not None else np.zeros(max(S, 1), dtype=np.int32)
    offs = out_offsets if out_offsets is not None else np.zeros(max(S, 1) + 1, dtype=np.int32)
    G, end, T = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    rc = L.lora_build_routing(n, p(slots), p(lens), S, p(perm), p(ids), p(offs), ctypes.byref(G),
                              ctypes.byref(end), ctypes.byref(T))
    _check(rc, "lora_build_routing")
    g = G.value
    keep_ids = ids[:g] if out_ids is not None else ids[:g].copy()
    keep_offs = offs[:g + 1] if out_offsets is not None else offs[:g + 1].copy()
    return {"perm": perm[:n].copy(), "lora_ids": keep_ids, "grouped_offsets": keep_offs,
            "num_groups": g, "end": end.value, "total_tokens": T.value}


def lora_build_token_rows(req_num_tokens, perm, end: int) -> np.ndarray:
    """Rows of the routed tokens in sorted order for an arrival-order batch."""
    L = lib()
    lens = np.ascontiguousarray(np.asarray(req_num_tokens, dtype=np.int32))
    pm = np.ascontiguousarray(np.asarray(perm, dtype=np.int32))
    out = np.zeros(max(int(end), 1), dtype=np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    _check(L.lora_build_token_rows(int(lens.size), p(lens), p(pm), int(end), p(out)), "lora_build_token_rows")
    return out[:int(end)].copy()


@dataclass
class Routing:
    """Routing triple: device lora_ids / grouped_offsets tensors, host num_groups / end,
    optionally device token_rows (row of each sorted token, unsorted batches),
    a host copy of grouped_offsets (int32 numpy array) that lets the library
    pick the kernels per group, and a host copy of lora_ids (with the host
    offsets: the mma.sync kernels take the triple as launch parameters)."""
    lora_ids: object
    grouped_offsets: object
    num_groups: int
    end: int
    token_rows: object = None
    host_grouped_offsets: object = None
    host_lora_ids: object = None

    def _c(self) -> _Routing:
        ptr = lambda t: t.data_ptr() if t is not None and t.numel() > 0 else None

        def host(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=np.int32)
            self._host_keep.append(a)  # the pointer must outlive the call
            return a.ctypes.data if a.size > 0 else None

        self._host_keep = []
        return _Routing(ptr(self.lora_ids), ptr(self.grouped_offsets), int(self.num_groups), int(self.end),
                        ptr(self.token_rows), host(self.host_grouped_offsets), host(self.host_lora_ids))


def routing_to_device(r: dict, device="cuda", non_blocking=False, host_offsets=False,
                      host_ids=False) -> Routing:
    """Upload the host triple from lora_build_routing (int32 tensors); with
    host_offsets the host copy of grouped_offsets rides along (per-group
    kernel choice), with host_ids also the host copy of lora_ids (the
    mma.sync kernels then take the triple as launch parameters)."""
    import torch
    ids_h = np.ascontiguousarray(r["lora_ids"], dtype=np.int32)[: int(r["num_groups"])]
    ids = torch.from_numpy(np.ascontiguousarray(r["lora_ids"], dtype=np.int32))
    offs_h = np.ascontiguousarray(r["grouped_offsets"], dtype=np.int32)
    offs = torch.from_numpy(offs_h)
    return Routing(ids.to(device, non_blocking=non_blocking), offs.to(device, non_blocking=non_blocking),
                   int(r["num_groups"]), int(r["end"]), None,
                   offs_h.copy() if host_offsets or host_ids else None, ids_h.copy() if host_ids else None)


# --------------------------------------------------------------- problems --

@dataclass
class Slice:
    """One projection slice: stacks A/B (device tensors), element offsets into
    them, slot strides, out_dim, and the output y (2-D tensor) with a column
    offset.  Row stride of y is taken from the tensor."""
    A: object
    A_slot_stride: int
    B: object
    B_slot_stride: int
    out_dim: int
    y: object
    A_offset: int = 0
    B_offset: int = 0
    y_col: int = 0
    bias: object = None          # optional [S, >= out] stack (element offset bias_offset)
    bias_slot_stride: int = 0
    bias_offset: int = 0


@dataclass
class Problem:
    x: object
    slices: List[Slice]
    max_num_loras: int
    max_lora_rank: int
    slot_ranks: object = None    # optional device int32 [S]: true ranks (skip the padding)
    _keep: list = field(default_factory=list)

    def _c(self) -> _Problem:
        import torch
        x = self.x
        if x.dim() != 2 or x.stride(1) != 1:
            raise ValueError("x must be 2-D with unit column stride")
        dt = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}.get(x.dtype)
        if dt is None:
            raise ValueError("x must be float32 or bfloat16")
        if not 1 <= len(self.slices) <= MAX_SLICES:
            raise ValueError("1..3 slices")
        es = x.element_size()
        arr = (_Slice * MAX_SLICES)()
        for j, s in enumerate(self.slices):
            for t in (s.A, s.B, s.y):
                if t.dtype != x.dtype:
                    raise ValueError("x, y, A and B must share one dtype")
            if s.y.dim() != 2 or s.y.stride(1) != 1:
                raise ValueError("y must be 2-D with unit column stride")
            bias_ptr = s.bias.data_ptr() + es * int(s.bias_offset) if s.bias is not None else None
            arr[j] = _Slice(s.A.data_ptr() + es * int(s.A_offset), int(s.A_slot_stride),
                            s.B.data_ptr() + es * int(s.B_offset), int(s.B_slot_stride), int(s.out_dim),
                            s.y.data_ptr() + es * int(s.y_col), int(s.y.stride(0)), bias_ptr,
                            int(s.bias_slot_stride))
        ranks = self.slot_ranks.data_ptr() if self.slot_ranks is not None else None
        return _Problem(dt, int(x.shape[0]), int(x.shape[1]), int(self.max_num_loras),
                        int(self.max_lora_rank), x.data_ptr(), int(x.stride(0)), len(self.slices), arr, ranks)


def fused_problem(x, A_fused, B_fused, y, out_dims: Sequence[int]) -> Problem:
    """Fused stacks A [S, n*R, in], B [S, O, R] and y [T, O] (QKV fusion: A on
    the rank dimension, B on the output dimension)."""
    S, nR, k = A_fused.shape
    n = len(out_dims)
    R = nR // n
    O = int(sum(out_dims))
    assert B_fused.shape == (S, O, R) and nR == n * R
    slices, off = [], 0
    for j, od in enumerate(out_dims):
        slices.append(Slice(A_fused, n * R * k, B_fused, O * R, int(od), y, A_offset=j * R * k,
                            B_offset=off * R, y_col=off))
        off += od
    return Problem(x, slices, S, R)


def per_projection_problem(x, A_list, B_list, y_list, y_cols=None) -> Problem:
    """Separate stacks per projection: A_j [S, R, in], B_j [S, out_j, R]; y_list
    gives each projection's output tensor (or one tensor repeated with y_cols)."""
    slices = []
    S, R, k = A_list[0].shape
    for j, (A, B, y) in enumerate(zip(A_list, B_list, y_list)):
        od = B.shape[1]
        slices.append(Slice(A, R * k, B, od * R, int(od), y, y_col=(y_cols[j] if y_cols else 0)))
    return Problem(x, slices, S, R)


# ---------------------------------------------------------------- calls --

def lora_set_slot(problem: Problem, slice_index: int, slot: int, r: int, lora_alpha: float,
                  use_rslora: bool, A_raw, B_raw, stream=None) -> None:
    import torch
    L = lib()
    raw_dt = DTYPE_BF16 if (A_raw is not None and A_raw.dtype == torch.bfloat16) else DTYPE_F32
    pa = A_raw.data_ptr() if A_raw is not None else None
    pb = B_raw.data_ptr() if B_raw is not None else None
    c = problem._c()
    _check(L.lora_set_slot(ctypes.byref(c), int(slice_index), int(slot), int(r), float(lora_alpha),
                           int(bool(use_rslora)), pa, pb, raw_dt, _stream_handle(stream)),
           "lora_set_slot")


def lora_set_slot_bias(problem: Problem, slice_index: int, slot: int, bias_raw, stream=None) -> None:
    import torch
    L = lib()
    raw_dt = DTYPE_BF16 if (bias_raw is not None and bias_raw.dtype == torch.bfloat16) else DTYPE_F32
    c = problem._c()
    _check(L.lora_set_slot_bias(ctypes.byref(c), int(slice_index), int(slot),
                                bias_raw.data_ptr() if bias_raw is not None else None, raw_dt,
                                _stream_handle(stream)), "lora_set_slot_bias")


def lora_shrink(problem: Problem, routing: Routing, u, stream=None) -> None:
    L = lib()
    c, rr = problem._c(), routing._c()
    _check(L.lora_shrink(ctypes.byref(c), ctypes.byref(rr), u.data_ptr() if u is not None else None,
                         _stream_handle(stream)), "lora_shrink")


def lora_expand(problem: Problem, routing: Routing, u, stream=None) -> None:
    L = lib()
    c, rr = problem._c(), routing._c()
    _check(L.lora_expand(ctypes.byref(c), ctypes.byref(rr), u.data_ptr() if u is not None else None,
                         _stream_handle(stream)), "lora_expand")


def lora_workspace_bytes(problem: Problem, end: int) -> int:
    c = problem._c()
    return int(lib().lora_workspace_bytes(ctypes.byref(c), int(end)))


def new_workspace(problem: Problem, end: int, device="cuda"):
    """A workspace tensor of lora_workspace_bytes(problem, end) bytes."""
    import torch
    nbytes = max(lora_workspace_bytes(problem, end), 256)
    return torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32, device=device)


def lora_sgmv_apply(problem: Problem, routing: Routing, workspace, stream=None) -> None:
    L = lib()
    c, rr = problem._c(), routing._c()
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(L.lora_sgmv_apply(ctypes.byref(c), ctypes.byref(rr),
                             workspace.data_ptr() if workspace is not None else None, nbytes,
                             _stream_handle(stream)), "lora_sgmv_apply")


def lora_base_gemm_apply(problem: Problem, routing: Routing, W0, workspace, stream=None) -> None:
    """The delta fused into the base projection: every row of each slice's
    y becomes W0_j x (+ the LoRA delta on routed rows), rounded once; y is
    written, not read.  W0: one device tensor [out_j, in] per slice (same
    dtype as x), or (tensor, element offset, row stride) tuples."""
    L = lib()
    c, rr = problem._c(), routing._c()
    arr = (_BaseWeight * MAX_SLICES)()
    if len(W0) != len(problem.slices):
        raise ValueError("one base weight per slice")
    for j, w in enumerate(W0):
        if isinstance(w, tuple):
            t, off, stride = w
        else:
            t, off, stride = w, 0, w.stride(0)
        if t.dtype != problem.x.dtype:
            raise ValueError("W0 must have the dtype of x")
        arr[j] = _BaseWeight(t.data_ptr() + t.element_size() * int(off), int(stride))
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(L.lora_base_gemm_apply(ctypes.byref(c), ctypes.byref(rr), arr,
                                  workspace.data_ptr() if workspace is not None else None, nbytes,
                                  _stream_handle(stream)), "lora_base_gemm_apply")


NOALLOC_MAX_WORKSPACE_BYTES = 16 * 1024 * 1024


def lora_sgmv_apply_noalloc(problem: Problem, routing: Routing, stream=None) -> None:
    """lora_sgmv_apply without a workspace argument, for callers that cannot
    allocate device memory: the intermediate lives in a fixed 16 MiB array
    inside the library.  Calls whose GPU work overlaps race on that array."""
    L = lib()
    c, rr = problem._c(), routing._c()
    _check(L.lora_sgmv_apply_noalloc(ctypes.byref(c), ctypes.byref(rr), _stream_handle(stream)),
           "lora_sgmv_apply_noalloc")


def lora_get_device_status(stream=None) -> int:
    L = lib()
    flags = ctypes.c_uint32(0)
    _check(L.lora_get_device_status(_stream_handle(stream), ctypes.byref(flags)),
           "lora_get_device_status")
    return int(flags.value)


def lora_last_call_path():
    """(path bits, kernel launches) of the most recent library call made on
    this host thread; see lora_last_call_path in include/lora_sgmv.h."""
    n = ctypes.c_uint32(0)
    bits = lib().lora_last_call_path(ctypes.byref(n))
    return int(bits), int(n.value)


def lora_selftest_wait_timeout(polls: int, stream=None) -> None:
    """Launch the failure-path self test: a bounded wait that runs out and
    sets LORA_DEV_TIMEOUT in the device status word (see include/lora_sgmv.h)."""
    _check(lib().lora_selftest_wait_timeout(int(polls), _stream_handle(stream)), "lora_selftest_wait_timeout")


def lora_status_string(status: int) -> str:
    return lib().lora_status_string(int(status)).decode()


class CallBuilder:
    """Pre-marshalled C arguments for repeated calls on fixed buffers (for
    CUDA-graph capture and the benchmark's hot loop): builds the ctypes
    structs once, then each call is a single foreign call."""

    def __init__(self, problem: Problem, routing: Routing, workspace):
        self.L = lib()
        self.c = problem._c()
        self.r = routing._c()
        self.ws = workspace.data_ptr()
        self.nbytes = workspace.numel() * workspace.element_size()
        self._keep = (problem, routing, workspace)
        self._n = ctypes.c_uint32(0)
        self.last_path = 0       # kernel families of the latest apply (lora_last_call_path)
        self.last_launches = 0   # kernels it launched

    def set_routing(self, num_groups: int, end: int) -> None:
        """A new batch in the same device routing buffers: only the host
        num_groups and end change."""
        self.r.num_groups = int(num_groups)
        self.r.end = int(end)

    def apply(self, stream=None) -> None:
        rc = self.L.lora_sgmv_apply(ctypes.byref(self.c), ctypes.byref(self.r), self.ws, self.nbytes,
                                    _stream_handle(stream))
        _check(rc, "lora_sgmv_apply")
        self.last_path = int(self.L.lora_last_call_path(ctypes.byref(self._n)))
        self.last_launches = int(self._n.value)
