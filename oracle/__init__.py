"""CPU oracle for the SGMV LoRA delta -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and this package shares no
code with the product: not the routing, not the weight preparation, not the
bf16 conversion.

What it computes, and where the pages define it:

* ``build_routing`` -- sort the batch so same-adapter requests are adjacent and
  base requests (slot -1) come last, then group consecutive same-adapter
  requests into ``(lora_ids, grouped_offsets, end)``, truncating at the first
  base group ("max.pipelines.lora.LoRAManagerV3" API page, sort_lora_batch and
  get_lora_graph_inputs).  Plain C in ``lora_oracle.c``.
* ``lora_scale`` -- scale = lora_alpha / r, or lora_alpha / sqrt(r) for rsLoRA
  ("vLLM LoRA 实现深度解析" section 1, the rsLoRA variant).
* ``prep_a`` / ``prep_b`` -- the load-time pipeline of the MAX page ("MAX
  max.pipelines.lora 模块解析", load pipeline: scale pre-multiplied into B, rank
  padding [r, in] -> [max_rank, in] and [out, r] -> [out, max_rank], dtype
  unification).  The scale is multiplied in fp32 and the product is rounded
  once to the storage type; this is what both pages' code does for fp32 and
  bf16 weights (numpy fp32 times a Python float; torch bf16 times a Python
  float computes in fp32 and rounds once).
* ``fuse_qkv_a`` / ``fuse_qkv_b`` -- QKV fusion: A concatenated on the rank
  dimension, B on the output dimension (same MAX page, QKV fusion).
* ``sgmv_rows`` -- the delta y_t += B_s . (A_s . x_t) for LoRA-routed rows,
  per slice, in double ("vLLM LoRA 实现深度解析" sections 1 and 6).  Plain C.

Storage types: ``"f32"`` arrays are numpy float32; ``"bf16"`` arrays are numpy
uint16 holding the bfloat16 bit pattern (the upper half of an IEEE binary32).
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_LIB = None
_LIB_OMP = None

OK, BAD_ARG, BAD_SLOT, BAD_ROW, BAD_ROUTE = 0, 1, 2, 3, 4


class _Slice(ctypes.Structure):
    _fields_ = [
        ("A", ctypes.c_void_p),
        ("A_slot_stride", ctypes.c_longlong),
        ("B", ctypes.c_void_p),
        ("B_slot_stride", ctypes.c_longlong),
        ("out_dim", ctypes.c_int),
        ("y_in", ctypes.c_void_p),
        ("y_in_row_stride", ctypes.c_longlong),
        ("y_out", ctypes.c_void_p),
        ("y_out_row_stride", ctypes.c_longlong),
        ("bias", ctypes.c_void_p),
        ("bias_slot_stride", ctypes.c_longlong),
    ]


def _bind(L):
    """Declare the oracle's C signatures on a loaded build."""
    i32p = ctypes.POINTER(ctypes.c_int)
    L.oracle_build_routing.restype = ctypes.c_int
    L.oracle_build_routing.argtypes = [ctypes.c_int, i32p, i32p, ctypes.c_int, i32p, i32p, i32p,
                                       i32p, i32p, i32p]
    L.oracle_sgmv_rows.restype = ctypes.c_int
    L.oracle_sgmv_rows.argtypes = [ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.POINTER(_Slice), ctypes.c_void_p,
                                   ctypes.c_longlong, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_void_p]
    L.oracle_base_rows.restype = ctypes.c_int
    L.oracle_base_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_longlong,
                                   ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_longlong]
    L.oracle_threads.restype = ctypes.c_int
    L.oracle_threads.argtypes = [ctypes.c_int]
    L.oracle_sgmv_token_slots.restype = ctypes.c_int
    L.oracle_sgmv_token_slots.argtypes = [ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(_Slice), ctypes.c_void_p,
                                          ctypes.c_longlong, ctypes.c_void_p]
    return L


def lib(parallel: bool = False):
    """Load (building first if needed) the C oracle: the single-threaded
    build, or with parallel=True the OpenMP build (bit-identical results;
    falls back to the single-threaded build where OpenMP is missing)."""
    global _LIB, _LIB_OMP
    if parallel:
        if _LIB_OMP is None:
            path = _build.omp_path()
            _LIB_OMP = _bind(ctypes.CDLL(path)) if path else lib(False)
        return _LIB_OMP
    if _LIB is None:
        _LIB = _bind(ctypes.CDLL(_build.build()))
    return _LIB


def omp_available() -> bool:
    return _build.omp_path() is not None


def threads(parallel: bool, n: int = 0) -> int:
    """Threads the (parallel or single-threaded) build runs its row loops on;
    n > 0 sets the OpenMP build's count first."""
    return int(lib(parallel).oracle_threads(int(n)))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


# --------------------------------------------------------------------------
# Storage-type conversions (exact decode; round-to-nearest-even encode)
# --------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact: bf16 is the top half of binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, IEEE round-to-nearest, ties to even.

    The discarded low 16 bits are compared with one half of the last kept
    bit; exact halves round to the even neighbour.  NaNs stay NaN (quiet bit
    set); infinities and overflow to infinity follow from the same rule.
    """
    a = np.ascontiguousarray(np.asarray(f, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    hi = u >> np.uint64(16)
    lo = u & np.uint64(0xFFFF)
    round_up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    out = (hi + round_up.astype(np.uint64)).astype(np.uint64)
    nan = np.isnan(a)
    out = np.where(nan, (hi | np.uint64(0x0040)), out)
    return out.astype(np.uint16)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored values to double."""
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    raise ValueError("unknown storage dtype %r" % (dtype,))


def from_f32(arr32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage type (one RNE rounding for bf16)."""
    if dtype == "bf16":
        return f32_to_bf16_bits(arr32)
    if dtype == "f32":
        return np.asarray(arr32, dtype=np.float32).copy()
    raise ValueError("unknown storage dtype %r" % (dtype,))


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

def build_routing(req_slot, req_len, max_num_loras: int) -> dict:
    """Sort + group into the routing triple (plain C; see lora_oracle.c)."""
    L = lib()
    slots = _i32(req_slot)
    lens = _i32(req_len)
    n = int(slots.size)
    S = int(max_num_loras)
    perm = np.zeros(max(n, 1), dtype=np.int32)
    ids = np.zeros(max(S, 1), dtype=np.int32)
    offs = np.zeros(S + 1, dtype=np.int32)
    G = ctypes.c_int(0)
    end = ctypes.c_int(0)
    T = ctypes.c_int(0)
    rc = L.oracle_build_routing(n, _p32(slots), _p32(lens), S, _p32(perm), _p32(ids), _p32(offs),
                                ctypes.byref(G), ctypes.byref(end), ctypes.byref(T))
    if rc != OK:
        return {"status": rc}
    g = G.value
    return {"status": OK, "perm": perm[:n].copy(), "lora_ids": ids[:g].copy(),
            "grouped_offsets": offs[:g + 1].copy(), "num_groups": g, "end": end.value,
            "total_tokens": T.value}


# --------------------------------------------------------------------------
# Load-time preparation (scale folding, rank padding, QKV fusion)
# --------------------------------------------------------------------------

def lora_scale(lora_alpha: float, r: int, use_rslora: bool) -> np.float32:
    """alpha / r, or alpha / sqrt(r) for rsLoRA; computed in double, kept as fp32."""
    if r <= 0:
        raise ValueError("rank must be positive")
    s = float(lora_alpha) / (math.sqrt(r) if use_rslora else float(r))
    return np.float32(s)


def prep_a(A_raw: np.ndarray, max_rank: int, dtype: str) -> np.ndarray:
    """[r, in] fp32 -> [max_rank, in] storage: rows >= r are zero."""
    A_raw = np.asarray(A_raw, dtype=np.float32)
    r, k = A_raw.shape
    if r > max_rank:
        raise ValueError("adapter rank %d exceeds max_lora_rank %d" % (r, max_rank))
    out = np.zeros((max_rank, k), dtype=np.float32)
    out[:r, :] = A_raw
    return from_f32(out, dtype)


def prep_b(B_raw: np.ndarray, max_rank: int, scale: np.float32, dtype: str) -> np.ndarray:
    """[out, r] fp32 -> scale folded in fp32 -> [out, max_rank] storage (cols >= r zero)."""
    B_raw = np.asarray(B_raw, dtype=np.float32)
    d, r = B_raw.shape
    if r > max_rank:
        raise ValueError("adapter rank %d exceeds max_lora_rank %d" % (r, max_rank))
    folded = (B_raw * np.float32(scale)).astype(np.float32)  # fp32 multiply, one rounding
    out = np.zeros((d, max_rank), dtype=np.float32)
    out[:, :r] = folded
    return from_f32(out, dtype)


def fuse_qkv_a(a_list):
    """Concatenate per-projection [R, in] A blocks on the rank dimension -> [n*R, in]."""
    return np.concatenate(list(a_list), axis=0)


def fuse_qkv_b(b_list):
    """Concatenate per-projection [out_j, R] B blocks on the output dimension -> [O, R]."""
    return np.concatenate(list(b_list), axis=0)


def lora_memory_bytes(num_lora_layers: int, in_features: int, out_features: int, rank: int,
                      dtype_bytes: int, max_loras: int) -> int:
    """GPU memory of the stacked A/B buffers ("vLLM LoRA 实现深度解析" section 9 formula)."""
    return num_lora_layers * (in_features * rank + out_features * rank) * dtype_bytes * max_loras


# --------------------------------------------------------------------------
# The delta
# --------------------------------------------------------------------------

def _bias_args(sl, keep):
    """(pointer, slot stride) of a slice's optional fp64 bias stack."""
    if sl.get("bias") is None:
        return None, 0
    b = np.ascontiguousarray(sl["bias"], dtype=np.float64)
    keep.append(b)
    return b.ctypes.data + 8 * int(sl.get("bias_offset", 0)), int(sl["bias_slot_stride"])


def sgmv_rows(rows, x_rows, slices, lora_ids, grouped_offsets, end: int, in_dim: int, R: int,
              max_num_loras: int, parallel: bool = False):
    """Delta for the listed rows, in double.

    rows           int array, batch row index of each listed row (< end)
    x_rows         float64 [n_rows, in_dim], the listed rows of x
    slices         list of dicts, one per projection slice:
                     A  float64 [S, >= R rows, in_dim] stack, or a flat view with
                        "A_slot_stride" (elements); rank row k of slot s at
                        A[s*A_slot_stride + k*in_dim : +in_dim]
                     B  float64 stack; element (s, o, k) at B[s*B_slot_stride + o*R + k]
                     out_dim, y_in float64 [n_rows, out_dim] (listed rows)
    parallel       use the OpenMP build (rows shared out among threads; the
                   same numbers)
    Returns (u [n_rows, n*R] float64, [y_out_j [n_rows, out_j] float64]).
    """
    L = lib(parallel)
    rows = _i32(rows)
    n = int(rows.size)
    x_rows = np.ascontiguousarray(x_rows, dtype=np.float64)
    assert x_rows.shape == (n, in_dim)
    ns = len(slices)
    keep = []
    arr = (_Slice * ns)()
    outs = []
    for j, sl in enumerate(slices):
        A = np.ascontiguousarray(sl["A"], dtype=np.float64)
        B = np.ascontiguousarray(sl["B"], dtype=np.float64)
        yi = np.ascontiguousarray(sl["y_in"], dtype=np.float64)
        od = int(sl["out_dim"])
        assert yi.shape == (n, od)
        yo = np.empty((n, od), dtype=np.float64)
        keep += [A, B, yi, yo]
        base_a = A.ctypes.data + 8 * int(sl.get("A_offset", 0))
        base_b = B.ctypes.data + 8 * int(sl.get("B_offset", 0))
        bias_ptr, bias_stride = _bias_args(sl, keep)
        arr[j] = _Slice(base_a, int(sl["A_slot_stride"]), base_b, int(sl["B_slot_stride"]), od,
                        yi.ctypes.data, od, yo.ctypes.data, od, bias_ptr, bias_stride)
        outs.append(yo)
    ids = _i32(lora_ids)
    offs = _i32(grouped_offsets)
    G = int(ids.size)
    assert offs.size == G + 1 or (G == 0 and offs.size >= 1)
    u = np.empty((n, ns * R), dtype=np.float64)
    rc = L.oracle_sgmv_rows(n, _p32(rows), int(in_dim), int(R), int(max_num_loras), ns, arr,
                            x_rows.ctypes.data, int(in_dim), _p32(ids), _p32(offs), G, int(end),
                            u.ctypes.data)
    if rc != OK:
        raise ValueError("oracle_sgmv_rows failed with code %d" % rc)
    return u, outs


def base_rows(W0, x_rows, parallel: bool = False):
    """The base projection W0 . x of the listed rows in double (plain C;
    W0 float64 [out, in], x_rows float64 [n, in]) -> float64 [n, out]."""
    W0 = np.ascontiguousarray(W0, dtype=np.float64)
    x_rows = np.ascontiguousarray(x_rows, dtype=np.float64)
    n, k = x_rows.shape
    out, k2 = W0.shape
    assert k == k2
    y = np.empty((n, out), dtype=np.float64)
    rc = lib(parallel).oracle_base_rows(n, k, out, W0.ctypes.data, k, x_rows.ctypes.data, k, y.ctypes.data, out)
    if rc != OK:
        raise ValueError("oracle_base_rows failed with code %d" % rc)
    return y


def prep_w0(W0_raw: np.ndarray, dtype: str) -> np.ndarray:
    """A base weight [out, in] (fp32) in the storage type (one RNE rounding)."""
    return from_f32(np.asarray(W0_raw, dtype=np.float32), dtype)


def problem_rows_with_base(prob, rows, W0_stored, parallel: bool = False):
    """The fused result for the listed rows: per slice j,
    y_j = W0_j . x_t + (t < end ? delta of t : 0)  (unrounded double), the
    base projection with the LoRA delta added (vLLM page section 1).
    W0_stored: one storage-type [out_j, in] weight per slice."""
    rows = _i32(rows)
    dt = prob["dtype"]
    x_rows = to_f64(prob["x"][rows], dt)
    bases = [base_rows(to_f64(w, dt), x_rows, parallel) for w in W0_stored]
    routed = rows < prob["end"]
    out = [b.copy() for b in bases]
    if routed.any():
        rr = rows[routed]
        slices = []
        for sl, b in zip(prob["slices"], bases):
            d = dict(sl)
            d["y_in"] = b[routed]
            slices.append(d)
        _, ys = sgmv_rows(rr, x_rows[routed], slices, prob["lora_ids"], prob["grouped_offsets"], prob["end"],
                          prob["in_dim"], prob["R"], prob["S"], parallel=parallel)
        for o, yj in zip(out, ys):
            o[routed] = yj
    return out


def problem_rows(prob, rows, parallel: bool = False):
    """Run ``sgmv_rows`` on a prepared problem (see ``prepare_problem``) for the given rows."""
    rows = _i32(rows)
    dt = prob["dtype"]
    x_rows = to_f64(prob["x"][rows], dt)
    slices = []
    for sl in prob["slices"]:
        d = dict(sl)
        d["y_in"] = to_f64(sl["y"][rows][:, sl["y_col0"]:sl["y_col0"] + sl["out_dim"]], dt)
        slices.append(d)
    return sgmv_rows(rows, x_rows, slices, prob["lora_ids"], prob["grouped_offsets"], prob["end"],
                     prob["in_dim"], prob["R"], prob["S"], parallel=parallel)


def prepare_problem(raw, proj: str, fused: bool = True) -> dict:
    """Oracle-side preparation of one projection problem from raw synthetic inputs.

    ``raw`` is a workload drawn by ``workloads.synthetic`` (raw fp32 adapter
    matrices per slot and projection, ranks, alphas, rsLoRA flags, request
    list, x and y in storage type).  ``proj`` is "qkv", "o", "gateup" or
    "down" (the last two: the MLP projections, gate + up fused).  Returns the
    routing (oracle's own), the stacked storage buffers and fp64 views.
    """
    dt = raw["dtype"]
    S, R = raw["max_num_loras"], raw["max_lora_rank"]
    names = {"qkv": ["q", "k", "v"], "o": ["o"], "gateup": ["gate", "up"], "down": ["down"]}[proj]
    route = build_routing(raw["req_slot"], raw["req_len"], S)
    in_dim = raw["x_" + proj].shape[1]
    outs = [raw["out_dims"][nm] for nm in names]
    stacks_a, stacks_b, stacks_bias = [], [], []
    has_bias = raw.get("bias") is not None
    for nm in names:
        if has_bias:  # the bias is added unscaled; stored in the storage type
            stacks_bias.append(np.stack([from_f32(np.asarray(raw["bias"][nm][s], dtype=np.float32), dt)
                                         for s in range(S)]))
        a_s, b_s = [], []
        for s in range(S):
            r = int(raw["rank"][s])
            sc = lora_scale(raw["alpha"][s], r, bool(raw["rslora"][s]))
            a_s.append(prep_a(raw["A"][nm][s], R, dt))
            b_s.append(prep_b(raw["B"][nm][s], R, sc, dt))
        stacks_a.append(np.stack(a_s))
        stacks_b.append(np.stack(b_s))
    slices = []
    y = raw["y_" + proj]
    if fused and len(names) > 1:
        A_st = np.stack([fuse_qkv_a([stacks_a[j][s] for j in range(len(names))]) for s in range(S)])
        B_st = np.stack([fuse_qkv_b([stacks_b[j][s] for j in range(len(names))]) for s in range(S)])
        A64, B64 = to_f64(A_st, dt), to_f64(B_st, dt)
        O = sum(outs)
        bias64 = to_f64(np.concatenate(stacks_bias, axis=1), dt) if has_bias else None
        off = 0
        for j, od in enumerate(outs):
            slices.append({"A": A64, "A_offset": j * R * in_dim, "A_slot_stride": len(names) * R * in_dim,
                           "B": B64, "B_offset": off * R, "B_slot_stride": O * R, "out_dim": od,
                           "y": y, "y_col0": off, "bias": bias64, "bias_offset": off, "bias_slot_stride": O})
            off += od
        stored = {"A": A_st, "B": B_st}
        if has_bias:
            stored["bias"] = np.concatenate(stacks_bias, axis=1)
    else:
        off = 0
        for j, od in enumerate(outs):
            slices.append({"A": to_f64(stacks_a[j], dt), "A_offset": 0, "A_slot_stride": R * in_dim,
                           "B": to_f64(stacks_b[j], dt), "B_offset": 0, "B_slot_stride": od * R,
                           "out_dim": od, "y": y, "y_col0": off,
                           "bias": to_f64(stacks_bias[j], dt) if has_bias else None, "bias_offset": 0,
                           "bias_slot_stride": od})
            off += od
        stored = {"A": stacks_a, "B": stacks_b} if len(names) > 1 else {"A": stacks_a[0], "B": stacks_b[0]}
        if has_bias:
            stored["bias"] = stacks_bias if len(names) > 1 else stacks_bias[0]
    return {"dtype": dt, "S": S, "R": R, "in_dim": in_dim, "x": raw["x_" + proj], "slices": slices,
            "lora_ids": route["lora_ids"], "grouped_offsets": route["grouped_offsets"],
            "end": route["end"], "route": route, "stored": stored, "out_dims": outs}


# --------------------------------------------------------------------------
# Unsorted batches: per-token slots
# --------------------------------------------------------------------------

def token_rows(req_len, perm, end: int) -> np.ndarray:
    """Rows (arrival-order batch) of the routed tokens in sorted order: the
    rows of request perm[0], then perm[1], ..., the first `end` of them."""
    lens = [int(v) for v in req_len]
    start = [0]
    for ln in lens:
        start.append(start[-1] + ln)
    out = []
    for i in perm:
        out.extend(range(start[int(i)], start[int(i)] + lens[int(i)]))
        if len(out) >= end:
            break
    return np.asarray(out[:end], dtype=np.int32)


def row_slots(req_slot, req_len) -> np.ndarray:
    """Slot of every row of an arrival-order batch (base -1): the per-token map."""
    return np.repeat(np.asarray(req_slot, dtype=np.int32), np.asarray(req_len, dtype=np.int64))


def sgmv_token_slots(row_slot, x_rows, slices, in_dim: int, R: int, max_num_loras: int,
                     parallel: bool = False):
    """Per-token definition (C): listed rows with their slots; see lora_oracle.c."""
    L = lib(parallel)
    rs = _i32(row_slot)
    n = int(rs.size)
    x_rows = np.ascontiguousarray(x_rows, dtype=np.float64)
    ns = len(slices)
    keep, arr, outs = [], (_Slice * ns)(), []
    for j, sl in enumerate(slices):
        A = np.ascontiguousarray(sl["A"], dtype=np.float64)
        B = np.ascontiguousarray(sl["B"], dtype=np.float64)
        yi = np.ascontiguousarray(sl["y_in"], dtype=np.float64)
        od = int(sl["out_dim"])
        yo = np.empty((n, od), dtype=np.float64)
        keep += [A, B, yi, yo]
        bias_ptr, bias_stride = _bias_args(sl, keep)
        arr[j] = _Slice(A.ctypes.data + 8 * int(sl.get("A_offset", 0)), int(sl["A_slot_stride"]),
                        B.ctypes.data + 8 * int(sl.get("B_offset", 0)), int(sl["B_slot_stride"]), od,
                        yi.ctypes.data, od, yo.ctypes.data, od, bias_ptr, bias_stride)
        outs.append(yo)
    u = np.empty((n, ns * R), dtype=np.float64)
    rc = L.oracle_sgmv_token_slots(n, _p32(rs), int(in_dim), int(R), int(max_num_loras), ns, arr,
                                   x_rows.ctypes.data, int(in_dim), u.ctypes.data)
    if rc != OK:
        raise ValueError("oracle_sgmv_token_slots failed with code %d" % rc)
    return u, outs


def problem_token_rows(prob, rows, row_slot, parallel: bool = False):
    """Per-token oracle on a prepared problem whose x / y are in arrival order."""
    rows = _i32(rows)
    dt = prob["dtype"]
    x_rows = to_f64(prob["x"][rows], dt)
    slices = []
    for sl in prob["slices"]:
        d = dict(sl)
        d["y_in"] = to_f64(sl["y"][rows][:, sl["y_col0"]:sl["y_col0"] + sl["out_dim"]], dt)
        slices.append(d)
    return sgmv_token_slots(row_slot, x_rows, slices, prob["in_dim"], prob["R"], prob["S"], parallel=parallel)
