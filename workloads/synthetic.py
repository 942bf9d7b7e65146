"""Seeded synthetic inputs for the SGMV LoRA workloads.

This module only DRAWS data: request lists, adapter ranks / alphas / rsLoRA
flags, raw (unscaled, unpadded) fp32 adapter matrices, and the activations x
and base outputs y in their storage type.  It holds none of the method's
arithmetic: no routing, no scale folding, no padding, no fusion, no delta.
Both the CUDA path and the CPU oracle are fed from here and each prepares its
own buffers.

Workload shapes (all attention projections; "hd" = head_dim):

  tiny        fp32; n_heads 8, n_kv 8, hd 16 (hidden 128, q/k/v 128 each);
              2 slots, max rank 16, ranks 4 and 8, alpha 8; requests with
              lengths [3,5,2,6,4] on adapters [0,0,1,1,base]
  decode8b    bf16; hidden 4096, n_heads 32, n_kv 8, hd 128 (q 4096, k/v 1024);
              8 slots, max rank 16, ranks from {8,16}; 256 one-token
              requests, 25% base, else uniform over the 8 slots
  prefill8b   bf16; same shapes; 4 slots plus base, max rank 64, ranks from
              {16,32,64}, alpha 2r, rsLoRA on 2 of the 4 slots; 16 requests
              with lengths uniform in [128, 2048], adapter uniform over
              {0,1,2,3,base}
  many64      bf16; 8B shapes; 64 slots, all rank 16; 1024 one-token
              requests, 10% base, else finite Zipf(s=1.1) over the 64 slots;
              per-projection (unfused) q/k/v plus o
  mixed64     bf16; 8B shapes; 64 slots, max rank 64, ranks from {16,32,64};
              3328 tokens = 4 prefill requests with lengths uniform in
              [512, 768] plus one-token decode requests for the rest; each
              request base with probability 0.1, else uniform over the slots
              (a few long groups among many short ones)
  mixed70b    bf16; hidden 8192, n_heads 64, n_kv 8, hd 128 (q 8192, k/v 1024);
              16 slots, max rank 128, ranks from {16,64,128}; 8192 tokens =
              6 prefill requests with lengths uniform in [512, 1024] plus
              one-token decode requests for the rest; each request base with
              probability 0.2, else uniform over the 16 slots

Values: x ~ N(0,1); A ~ N(0,1)/sqrt(in); B ~ 0.02 N(0,1) (raw, before the
scale is folded in); y ~ N(0,1) (the base projection's output).  Where a
workload leaves lora_alpha open it is 2r.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

PROJS = ("q", "k", "v", "o")
MLP_PROJS = ("gate", "up", "down")
# Problems of a layer: one shared input per problem, its projections as slices.
PROBLEMS = {"qkv": ("q", "k", "v"), "o": ("o",), "gateup": ("gate", "up"), "down": ("down",)}


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    dtype: str                     # "f32" or "bf16" (storage type of x, y, A, B)
    n_heads: int
    n_kv_heads: int
    head_dim: int
    hidden: int
    max_num_loras: int
    max_lora_rank: int
    rank_choices: Sequence[int]
    alpha_rule: str = "2r"         # "2r" or a fixed number as a string, e.g. "8"
    rslora_count: int = 0          # number of slots (drawn by the rng) using rsLoRA
    fused_qkv: bool = True
    # request list
    kind: str = "decode"           # "fixed", "decode", "prefill", "mixed", "custom"
    n_requests: int = 0
    base_prob: float = 0.0
    slot_dist: str = "uniform"     # "uniform", "uniform+base" (base is one more choice), "zipf1.1"
    len_range: Sequence[int] = (1, 1)
    total_tokens: int = 0
    n_prefill: int = 0
    fixed_slots: Optional[Sequence[int]] = None
    fixed_lens: Optional[Sequence[int]] = None
    fixed_ranks: Optional[Sequence[int]] = None
    family: str = "attn"           # "attn": q/k/v + o; "mlp": gate/up + down
    intermediate: int = 0          # MLP intermediate width

    @property
    def projs(self):
        return MLP_PROJS if self.family == "mlp" else PROJS

    @property
    def problems(self):
        return ("gateup", "down") if self.family == "mlp" else ("qkv", "o")

    @property
    def out_dims(self):
        if self.family == "mlp":
            return {"gate": self.intermediate, "up": self.intermediate, "down": self.hidden}
        q = self.n_heads * self.head_dim
        kv = self.n_kv_heads * self.head_dim
        return {"q": q, "k": kv, "v": kv, "o": self.hidden}

    @property
    def in_dims(self):
        if self.family == "mlp":
            return {"gate": self.hidden, "up": self.hidden, "down": self.intermediate}
        return {"q": self.hidden, "k": self.hidden, "v": self.hidden,
                "o": self.n_heads * self.head_dim}


SPECS = {
    "tiny": Spec("tiny", "f32", 8, 8, 16, 128, 2, 16, (4, 8), alpha_rule="8", kind="fixed",
                 fixed_slots=(0, 0, 1, 1, -1), fixed_lens=(3, 5, 2, 6, 4), fixed_ranks=(4, 8)),
    "decode8b": Spec("decode8b", "bf16", 32, 8, 128, 4096, 8, 16, (8, 16), kind="decode",
                     n_requests=256, base_prob=0.25, slot_dist="uniform"),
    "prefill8b": Spec("prefill8b", "bf16", 32, 8, 128, 4096, 4, 64, (16, 32, 64), rslora_count=2,
                      kind="prefill", n_requests=16, slot_dist="uniform+base", len_range=(128, 2048)),
    "many64": Spec("many64", "bf16", 32, 8, 128, 4096, 64, 16, (16,), fused_qkv=False, kind="decode",
                   n_requests=1024, base_prob=0.10, slot_dist="zipf1.1"),
    "mixed70b": Spec("mixed70b", "bf16", 64, 8, 128, 8192, 16, 128, (16, 64, 128), kind="mixed",
                     total_tokens=8192, n_prefill=6, base_prob=0.20, slot_dist="uniform",
                     len_range=(512, 1024)),
    # A mixed batch over many adapters: a few long prefill segments among
    # many one-token decode groups (the kernels are then picked per group).
    "mixed64": Spec("mixed64", "bf16", 32, 8, 128, 4096, 64, 64, (16, 32, 64), kind="mixed",
                    total_tokens=3328, n_prefill=4, base_prob=0.10, slot_dist="uniform",
                    len_range=(512, 768)),
    # MLP projections of the same 8B shape (intermediate 14336): gate + up
    # fused as a two-slice problem, down separately.
    "mlp8b": Spec("mlp8b", "bf16", 32, 8, 128, 4096, 8, 16, (8, 16), kind="decode",
                  n_requests=256, base_prob=0.25, slot_dist="uniform", family="mlp",
                  intermediate=14336),
}


def _slot_draw(rng, spec: Spec, n: int) -> np.ndarray:
    S = spec.max_num_loras
    if spec.slot_dist == "uniform+base":
        c = rng.integers(0, S + 1, size=n)
        return np.where(c == S, -1, c).astype(np.int32)
    if spec.slot_dist == "uniform":
        s = rng.integers(0, S, size=n)
    elif spec.slot_dist == "zipf1.1":
        k = np.arange(1, S + 1, dtype=np.float64)
        p = k ** -1.1
        p /= p.sum()
        s = rng.choice(S, size=n, p=p)
    else:
        raise ValueError(spec.slot_dist)
    base = rng.random(n) < spec.base_prob
    return np.where(base, -1, s).astype(np.int32)


def draw_requests(rng, spec: Spec):
    """Request list in arrival order: (slot per request, tokens per request)."""
    if spec.kind == "fixed":
        return (np.asarray(spec.fixed_slots, dtype=np.int32),
                np.asarray(spec.fixed_lens, dtype=np.int32))
    if spec.kind == "decode":
        n = spec.n_requests
        return _slot_draw(rng, spec, n), np.ones(n, dtype=np.int32)
    if spec.kind == "prefill":
        n = spec.n_requests
        lens = rng.integers(spec.len_range[0], spec.len_range[1] + 1, size=n).astype(np.int32)
        return _slot_draw(rng, spec, n), lens
    if spec.kind == "mixed":
        lens_p = rng.integers(spec.len_range[0], spec.len_range[1] + 1,
                              size=spec.n_prefill).astype(np.int32)
        n_dec = spec.total_tokens - int(lens_p.sum())
        lens = np.concatenate([lens_p, np.ones(n_dec, dtype=np.int32)])
        return _slot_draw(rng, spec, lens.size), lens
    raise ValueError(spec.kind)


def to_storage(a32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 numpy -> storage type (bf16 as uint16 bit patterns, via torch's cast)."""
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def draw(spec, seed: int = 0, with_weights: bool = True, requests=None) -> dict:
    """Draw one workload instance.  Deterministic in (spec, seed, requests).

    requests=(slots, lens) reuses another instance's request list (another
    layer of the same batch): adapters, x and y are still drawn from `seed`."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    rng = np.random.default_rng(seed)
    if requests is None:
        slots, lens = draw_requests(rng, spec)
    else:
        slots = np.asarray(requests[0], dtype=np.int32).copy()
        lens = np.asarray(requests[1], dtype=np.int32).copy()
    S, R = spec.max_num_loras, spec.max_lora_rank
    if spec.fixed_ranks is not None:
        ranks = np.asarray(spec.fixed_ranks, dtype=np.int32)
    else:
        ranks = rng.choice(np.asarray(spec.rank_choices, dtype=np.int32), size=S).astype(np.int32)
    if spec.alpha_rule == "2r":
        alphas = (2.0 * ranks).astype(np.float64)
    else:
        alphas = np.full(S, float(spec.alpha_rule))
    rslora = np.zeros(S, dtype=bool)
    if spec.rslora_count:
        rslora[rng.choice(S, size=spec.rslora_count, replace=False)] = True
    T = int(lens.sum())
    out = {"spec": spec, "seed": seed, "dtype": spec.dtype, "max_num_loras": S, "max_lora_rank": R,
           "req_slot": slots, "req_len": lens, "T": T, "rank": ranks, "alpha": alphas,
           "rslora": rslora, "out_dims": spec.out_dims, "in_dims": spec.in_dims,
           "fused_qkv": spec.fused_qkv}
    if with_weights:
        A, B = {}, {}
        for p in spec.projs:
            kin, dout = spec.in_dims[p], spec.out_dims[p]
            A[p], B[p] = [], []
            for s in range(S):
                r = int(ranks[s])
                A[p].append(rng.standard_normal((r, kin), dtype=np.float32) / np.float32(np.sqrt(kin)))
                B[p].append(np.float32(0.02) * rng.standard_normal((dout, r), dtype=np.float32))
        out["A"], out["B"] = A, B
    out["problems"] = spec.problems
    for prob in spec.problems:
        names = PROBLEMS[prob]
        k_in = spec.in_dims[names[0]]
        O = sum(spec.out_dims[p] for p in names)
        out["x_" + prob] = to_storage(rng.standard_normal((T, k_in), dtype=np.float32), spec.dtype)
    for prob in spec.problems:
        O = sum(spec.out_dims[p] for p in PROBLEMS[prob])
        out["y_" + prob] = to_storage(rng.standard_normal((T, O), dtype=np.float32), spec.dtype)
    return out


def custom_spec(**kw) -> Spec:
    """A Spec for tests: any field of Spec may be overridden; name defaults to "custom"."""
    base = dict(name="custom", dtype="bf16", n_heads=4, n_kv_heads=2, head_dim=32, hidden=128,
                max_num_loras=4, max_lora_rank=16, rank_choices=(8, 16), kind="decode",
                n_requests=8, base_prob=0.2, slot_dist="uniform")
    base.update(kw)
    return Spec(**base)


def emphasize_delta(raw: dict, b_factor: float = 40.0) -> dict:
    """A variant of a drawn workload whose check is dominated by the LoRA
    delta: every base output y is zero and the raw B matrices are multiplied
    by b_factor (B ~ 0.02 * b_factor * N(0, 1) before the scale is folded in,
    so the delta is of order one or more instead of about 0.1).  Only the
    drawn data change; no part of the method is applied here."""
    spec = raw["spec"]
    for prob in spec.problems:
        raw["y_" + prob] = to_storage(np.zeros(raw["y_" + prob].shape, dtype=np.float32), spec.dtype)
    for p in spec.projs:
        raw["B"][p] = [np.float32(b_factor) * b for b in raw["B"][p]]
    return raw


def add_base_weights(raw: dict, seed: int = 0) -> dict:
    """Draw the base projection weights W0 [out, in] per projection, fp32,
    N(0, 1) / sqrt(in) (the projection the LoRA delta is added to), from
    their own stream so the rest of the workload is unchanged."""
    rng = np.random.default_rng([seed, 104729])
    spec = raw["spec"]
    raw["W0"] = {p: rng.standard_normal((spec.out_dims[p], spec.in_dims[p]), dtype=np.float32)
                 / np.float32(np.sqrt(spec.in_dims[p])) for p in spec.projs}
    return raw


def add_bias(raw: dict, seed: int = 0, scale: float = 0.1) -> dict:
    """Draw a LoRA bias vector per (projection, slot): scale * N(0, 1), fp32.
    Drawn from its own stream so the rest of the workload is unchanged."""
    rng = np.random.default_rng([seed, 7919])
    spec = raw["spec"]
    raw["bias"] = {p: [np.float32(scale) * rng.standard_normal(spec.out_dims[p], dtype=np.float32)
                       for _ in range(spec.max_num_loras)] for p in spec.projs}
    return raw
