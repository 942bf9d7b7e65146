"""Device buffers for a drawn synthetic workload, built through the library.

Given raw inputs from ``workloads.synthetic.draw`` this allocates the device
tensors (x, y, stacked A/B, workspace) with torch and fills the stacks by
calling the library's own ``lora_set_slot`` once per (slot, slice); routing
comes from the library's ``lora_build_routing``.  Nothing here computes any
part of the method: it is allocation, upload and calls into the product.
"""
from __future__ import annotations

import numpy as np
import torch

import adapter_sgmv_lora_gb300 as lk

_TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def storage_to_torch(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Storage array (bf16 bits as uint16, or float32) -> device tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


def torch_to_storage(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def prepare(raw: dict, proj: str, fused: bool = True, device="cuda", separate_y: bool = False,
            slot_ranks: bool = False, shared_routing=None, host_offsets: bool = False,
            host_ids: bool = False) -> dict:
    """Build one projection problem ("qkv", "o", "gateup" or "down") on the device.

    fused=True: one fused stack A [S, n*R, in], B [S, O, R] and y [T, O].
    fused=False: per-projection stacks A_j [S, R, in], B_j [S, out_j, R]; y is
    one [T, O] tensor addressed by column offsets, or (separate_y) one tensor
    per projection.  When the workload carries a bias (synthetic.add_bias) the
    slices get bias stacks filled by lora_set_slot_bias; slot_ranks=True
    passes the slots' true ranks so the kernels skip the padding.
    shared_routing=(route_host, routing) reuses another problem's routing (the
    same batch): no new triple is built or uploaded.  host_offsets=True gives
    the routing its host copy of grouped_offsets (kernels picked per group);
    host_ids=True adds the host copy of lora_ids too (the mma.sync kernels
    take the whole triple as launch parameters).
    """
    dt = raw["dtype"]
    tdt = _TORCH_DT[dt]
    S, R = raw["max_num_loras"], raw["max_lora_rank"]
    from workloads.synthetic import PROBLEMS
    names = list(PROBLEMS[proj])
    outs = [raw["out_dims"][nm] for nm in names]
    O = sum(outs)
    x = storage_to_torch(raw["x_" + proj], dt, device)
    T, k = x.shape
    y_all = storage_to_torch(raw["y_" + proj], dt, device)
    has_bias = raw.get("bias") is not None
    if fused or len(names) == 1:
        A = torch.empty((S, len(names) * R, k), dtype=tdt, device=device)
        B = torch.empty((S, O, R), dtype=tdt, device=device)
        prob = lk.fused_problem(x, A, B, y_all, outs)
        stacks = {"A": A, "B": B}
        if has_bias:
            bias = torch.empty((S, O), dtype=tdt, device=device)
            off = 0
            for sl, od in zip(prob.slices, outs):
                sl.bias, sl.bias_slot_stride, sl.bias_offset = bias, O, off
                off += od
            stacks["bias"] = bias
        ys = [y_all]
    else:
        As = [torch.empty((S, R, k), dtype=tdt, device=device) for _ in names]
        Bs = [torch.empty((S, od, R), dtype=tdt, device=device) for od in outs]
        if separate_y:
            cols = np.cumsum([0] + outs)
            ys = [y_all[:, cols[j]:cols[j + 1]].contiguous() for j in range(len(names))]
            prob = lk.per_projection_problem(x, As, Bs, ys)
        else:
            cols = list(np.cumsum([0] + outs)[:-1])
            ys = [y_all]
            prob = lk.per_projection_problem(x, As, Bs, [y_all] * len(names), y_cols=cols)
        stacks = {"A": As, "B": Bs}
        if has_bias:
            stacks["bias"] = []
            for sl, od in zip(prob.slices, outs):
                sl.bias, sl.bias_slot_stride = torch.empty((S, od), dtype=tdt, device=device), od
                stacks["bias"].append(sl.bias)
    if slot_ranks:
        prob.slot_ranks = torch.from_numpy(np.asarray(raw["rank"], dtype=np.int32)).to(device)
    for j, nm in enumerate(names):
        for s in range(S):
            r = int(raw["rank"][s])
            a_raw = torch.from_numpy(np.ascontiguousarray(raw["A"][nm][s], dtype=np.float32)).to(device)
            b_raw = torch.from_numpy(np.ascontiguousarray(raw["B"][nm][s], dtype=np.float32)).to(device)
            lk.lora_set_slot(prob, j, s, r, float(raw["alpha"][s]), bool(raw["rslora"][s]), a_raw, b_raw)
            if has_bias:
                bias_raw = torch.from_numpy(np.ascontiguousarray(raw["bias"][nm][s], dtype=np.float32)).to(device)
                lk.lora_set_slot_bias(prob, j, s, bias_raw)
    if shared_routing is None:
        rt = lk.lora_build_routing(raw["req_slot"], raw["req_len"], S)
        routing = lk.routing_to_device(rt, device, host_offsets=host_offsets, host_ids=host_ids)
    else:
        rt, routing = shared_routing
    ws = lk.new_workspace(prob, rt["end"], device=device)
    return {"problem": prob, "routing": routing, "route_host": rt, "x": x, "ys": ys, "y_all": y_all,
            "stacks": stacks, "workspace": ws, "dtype": dt, "names": names, "outs": outs,
            "separate_y": (not fused and separate_y and len(names) > 1)}


def y_host(dev: dict) -> np.ndarray:
    """The problem's y as one [T, O] storage array (concatenating separate outputs)."""
    if dev["separate_y"]:
        return np.concatenate([torch_to_storage(y, dev["dtype"]) for y in dev["ys"]], axis=1)
    return torch_to_storage(dev["y_all"], dev["dtype"])
