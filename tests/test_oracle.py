"""Pins for the CPU oracle: it is checked against what the pages and the
mathematics fix, never against itself or the CUDA path.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, an unstable sort, a wrong scale)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import synthetic as sy

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- routing --

@pytest.mark.parametrize("name", ["routing_tiny.json", "routing_unsorted.json"])
def test_routing_golden(name):
    g = _gold(name)
    r = oracle.build_routing(g["req_slot"], g["req_len"], g["max_num_loras"])
    assert r["status"] == oracle.OK
    assert r["perm"].tolist() == g["perm"]
    assert r["lora_ids"].tolist() == g["lora_ids"]
    assert r["grouped_offsets"].tolist() == g["grouped_offsets"]
    assert r["num_groups"] == g["num_groups"]
    assert r["end"] == g["end"]
    assert r["total_tokens"] == g["total_tokens"]


def _token_slots_naive(slots, lens, perm):
    """Slot of every token row of the sorted batch, base rows as -1."""
    out = []
    for i in perm:
        out += [int(slots[i])] * int(lens[i])
    return out


def _token_slots_from_triple(r, T):
    out = [-1] * T
    for g in range(r["num_groups"]):
        for t in range(r["grouped_offsets"][g], r["grouped_offsets"][g + 1]):
            out[t] = int(r["lora_ids"][g])
    return out


def test_routing_brute_force():
    """Every slot assignment of up to 5 requests over 3 slots plus base, with
    lengths including 0: perm matches Python's stable sort, and the triple
    expands to exactly the naive per-token slot map of the sorted batch."""
    rng = np.random.default_rng(1)
    S = 3
    n_cases = 0
    for n in range(0, 6):
        for slots in itertools.product(range(-1, S), repeat=n):
            lens = rng.integers(0, 4, size=n).astype(np.int32)
            r = oracle.build_routing(list(slots), lens, S)
            assert r["status"] == oracle.OK
            key = lambda i: (slots[i] < 0, slots[i])
            perm = sorted(range(n), key=key)  # Python's sort is stable
            assert r["perm"].tolist() == perm
            T = int(lens.sum())
            assert r["total_tokens"] == T
            naive = _token_slots_naive(slots, lens, perm)
            # every row before the first base row is routed; base rows are last
            assert _token_slots_from_triple(r, T) == naive
            offs = r["grouped_offsets"]
            assert offs[0] == 0 and offs[-1] == r["end"]
            assert np.all(np.diff(offs) >= 0)
            ids = r["lora_ids"].tolist()
            assert len(set(ids)) == len(ids) <= S
            assert ids == sorted(ids)
            assert r["end"] == int(sum(l for s, l in zip(slots, lens) if s >= 0))
            n_cases += 1
    assert n_cases == sum(4 ** n for n in range(6))


def test_routing_errors():
    assert oracle.build_routing([0, 3], [1, 1], 3)["status"] == oracle.BAD_SLOT
    assert oracle.build_routing([-2], [1], 3)["status"] == oracle.BAD_SLOT
    assert oracle.build_routing([0], [-1], 3)["status"] == oracle.BAD_ARG
    r = oracle.build_routing([], [], 4)
    assert r["status"] == oracle.OK and r["num_groups"] == 0 and r["end"] == 0


def test_routing_all_base_and_empty_groups():
    r = oracle.build_routing([-1, -1], [3, 2], 2)
    assert r["num_groups"] == 0 and r["end"] == 0 and r["total_tokens"] == 5
    r = oracle.build_routing([1, 0, 1], [0, 2, 0], 2)
    assert r["lora_ids"].tolist() == [0, 1]
    assert r["grouped_offsets"].tolist() == [0, 2, 2]


# ----------------------------------------------------------- conversions --

def test_bf16_rounding_pins():
    f = np.array([1.0, -0.0, np.inf, -np.inf], dtype=np.float32)
    assert oracle.f32_to_bf16_bits(f).tolist() == [0x3F80, 0x8000, 0x7F80, 0xFF80]
    bits = np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF, 0x7F7FFFFF], dtype=np.uint32)
    got = oracle.f32_to_bf16_bits(bits.view(np.float32)).tolist()
    # tie to even (down), tie to even (up), above half, below half, overflow to inf
    assert got == [0x3F80, 0x3F82, 0x3F81, 0x3F80, 0x7F80]
    nan = oracle.f32_to_bf16_bits(np.array([np.nan], dtype=np.float32))
    assert np.isnan(oracle.bf16_bits_to_f32(nan))[0]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    f = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # plant exact ties
    u = f.view(np.uint32).copy()
    u[::7] = (u[::7] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    f = u.view(np.float32)
    mine = oracle.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    back = oracle.bf16_bits_to_f32(mine)
    assert np.array_equal(back, torch.from_numpy(f).to(torch.bfloat16).float().numpy())


# ----------------------------------------------------------------- scale --

def test_scale_page_numbers():
    p = _gold("page_numbers.json")
    e = p["scale_example"]
    assert oracle.lora_scale(e["lora_alpha"], e["r"], False) == np.float32(e["scaling"])
    e = p["rslora_example"]
    assert oracle.lora_scale(e["lora_alpha"], e["r"], True) == np.float32(e["scaling"])
    e = p["tiny_adapter_scales"]
    assert [float(oracle.lora_scale(e["lora_alpha"], r, False)) for r in e["ranks"]] == e["scaling"]
    e = p["memory_formula"]
    assert oracle.lora_memory_bytes(e["num_lora_layers"], e["in_features"], e["out_features"],
                                    e["rank"], e["dtype_bytes"], e["max_loras"]) == e["bytes"]
    assert oracle.lora_scale(16, 9, True) == np.float32(16 / 3)


def test_prep_shapes_and_padding():
    rng = np.random.default_rng(3)
    A = rng.standard_normal((4, 10)).astype(np.float32)
    B = rng.standard_normal((6, 4)).astype(np.float32)
    a = oracle.prep_a(A, 16, "f32")
    b = oracle.prep_b(B, 16, np.float32(0.5), "f32")
    assert a.shape == (16, 10) and b.shape == (6, 16)
    assert np.array_equal(a[:4], A) and not a[4:].any()
    assert np.array_equal(b[:, :4], B * np.float32(0.5)) and not b[:, 4:].any()
    with pytest.raises(ValueError):
        oracle.prep_a(A, 3, "f32")
    ab = oracle.prep_b(B, 8, np.float32(3.0), "bf16")
    # scale in fp32, then one cast to the storage type (MAX load pipeline order)
    ref = (torch.from_numpy(B) * torch.tensor(3.0, dtype=torch.float32)).to(torch.bfloat16)
    assert np.array_equal(oracle.bf16_bits_to_f32(ab[:, :4]), ref.float().numpy())


# ----------------------------------------------------------------- delta --

def _worked():
    g = _gold("worked_delta.json")
    R, S, k = g["max_lora_rank"], g["max_num_loras"], g["in_dim"]
    A = np.zeros((S, R, k))
    B = np.zeros((S, 3, R))
    for s in range(S):
        sc = oracle.lora_scale(g["alpha"][s], g["rank"][s], False)
        A[s] = oracle.prep_a(np.array(g["A_raw"][s], dtype=np.float32), R, "f32")
        B[s] = oracle.prep_b(np.array(g["B_raw"][s], dtype=np.float32), R, sc, "f32")
    return g, A, B


def test_worked_example_golden():
    g, A, B = _worked()
    x = np.array(g["x"], dtype=np.float64)
    yi = np.array(g["y_in"], dtype=np.float64)
    rows = [0, 1]
    sl = [{"A": A, "A_slot_stride": A.shape[1] * A.shape[2], "B": B, "B_slot_stride": 3 * 2,
           "out_dim": 3, "y_in": yi[rows]}]
    u, (yo,) = oracle.sgmv_rows(rows, x[rows], sl, g["lora_ids"], g["grouped_offsets"], g["end"],
                                3, 2, 2)
    assert u.tolist() == g["u"]
    assert yo.tolist() == g["y_out"][:2]
    # the base row (row 2 >= end) is never produced
    with pytest.raises(ValueError):
        oracle.sgmv_rows([2], x[[2]], [dict(sl[0], y_in=yi[[2]])], g["lora_ids"],
                         g["grouped_offsets"], g["end"], 3, 2, 2)


def _rand_problem(rng, S=3, R=8, k=24, outs=(16, 8, 8), ranks=None, T=12):
    ranks = ranks or [R] * S
    A = [np.zeros((S, R, k)) for _ in outs]
    B = [np.zeros((S, o, R)) for o in outs]
    Araw, Braw = [], []
    for j, o in enumerate(outs):
        Araw.append([]), Braw.append([])
        for s in range(S):
            a = rng.standard_normal((ranks[s], k))
            b = rng.standard_normal((o, ranks[s]))
            A[j][s, :ranks[s]] = a
            B[j][s, :, :ranks[s]] = b
            Araw[j].append(a), Braw[j].append(b)
    x = rng.standard_normal((T, k))
    ys = [rng.standard_normal((T, o)) for o in outs]
    return A, B, Araw, Braw, x, ys


def _slices(A, B, ys, rows, R, k):
    return [{"A": A[j], "A_slot_stride": R * k, "B": B[j], "B_slot_stride": B[j].shape[1] * R,
             "out_dim": B[j].shape[1], "y_in": ys[j][rows]} for j in range(len(A))]


def test_merged_weight_brute_force():
    """y_out = (W0 + B_s A_s) x for y_in = W0 x: the delta is the merged-weight
    product, computed here by numpy matmul in double."""
    rng = np.random.default_rng(4)
    S, R, k, outs, T = 3, 8, 24, (16, 8, 8), 12
    A, B, _, _, x, _ = _rand_problem(rng, S, R, k, outs, ranks=[5, 8, 3], T=T)
    W0 = [rng.standard_normal((o, k)) for o in outs]
    ys = [x @ W.T for W in W0]
    lora_ids, offs, end = [2, 0, 1], [0, 3, 7, 10], 10
    rows = list(range(end))
    u, yo = oracle.sgmv_rows(rows, x[rows], _slices(A, B, ys, rows, R, k), lora_ids, offs, end,
                             k, R, S)
    for j in range(len(outs)):
        for g in range(3):
            s = lora_ids[g]
            W = W0[j] + B[j][s] @ A[j][s]
            for t in range(offs[g], offs[g + 1]):
                ref = W @ x[t]
                np.testing.assert_allclose(yo[j][t], ref, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(u[t, j * R:(j + 1) * R], A[j][s] @ x[t], rtol=1e-12,
                                           atol=1e-12)


def test_zero_b_leaves_y_unchanged():
    """The pages' toy adapter has B = 0: y must come back exactly as it went in."""
    rng = np.random.default_rng(5)
    A, B, _, _, x, ys = _rand_problem(rng)
    B = [np.zeros_like(b) for b in B]
    rows = list(range(10))
    _, yo = oracle.sgmv_rows(rows, x[rows], _slices(A, B, ys, rows, 8, 24), [2, 0, 1],
                             [0, 3, 7, 10], 10, 24, 8, 3)
    for j in range(3):
        assert np.array_equal(yo[j], ys[j][rows])


def test_rank_padding_changes_nothing():
    """Zero-padding A rows / B columns from r to max_rank adds only exact zeros."""
    rng = np.random.default_rng(6)
    S, k, r = 2, 20, 5
    A = rng.standard_normal((S, r, k))
    B = rng.standard_normal((S, 7, r))
    x = rng.standard_normal((6, k))
    y = rng.standard_normal((6, 7))
    rows = list(range(6))
    args = ([1, 0], [0, 2, 6], 6)
    sl = [{"A": A, "A_slot_stride": r * k, "B": B, "B_slot_stride": 7 * r, "out_dim": 7,
           "y_in": y}]
    u1, (y1,) = oracle.sgmv_rows(rows, x, sl, *args, k, r, S)
    for Rp in (8, 16):
        Ap = np.zeros((S, Rp, k)); Ap[:, :r] = A
        Bp = np.zeros((S, 7, Rp)); Bp[:, :, :r] = B
        slp = [{"A": Ap, "A_slot_stride": Rp * k, "B": Bp, "B_slot_stride": 7 * Rp, "out_dim": 7,
                "y_in": y}]
        u2, (y2,) = oracle.sgmv_rows(rows, x, slp, *args, k, Rp, S)
        assert np.array_equal(y1, y2)
        assert np.array_equal(u1, u2[:, :r]) and not u2[:, r:].any()


def test_slot_routing_picks_the_right_adapter():
    """Each group uses its own slot: swapping lora_ids swaps the results."""
    rng = np.random.default_rng(7)
    A, B, _, _, x, ys = _rand_problem(rng, T=6)
    rows = list(range(6))
    sl = _slices(A, B, ys, rows, 8, 24)
    _, ya = oracle.sgmv_rows(rows, x, sl, [0, 1], [0, 3, 6], 6, 24, 8, 3)
    _, yb = oracle.sgmv_rows(rows, x, sl, [1, 0], [0, 3, 6], 6, 24, 8, 3)
    _, yc = oracle.sgmv_rows(rows, x, sl, [1, 1], [0, 3, 6], 6, 24, 8, 3)
    assert not np.allclose(ya[0][:3], yb[0][:3])
    assert np.array_equal(yb[0][:3], yc[0][:3])
    assert np.array_equal(ya[0][3:], yc[0][3:])


def test_homogeneity():
    """Doubling x doubles the delta exactly (power-of-two scaling is exact)."""
    rng = np.random.default_rng(8)
    A, B, _, _, x, ys = _rand_problem(rng)
    rows = list(range(10))
    zeros = [np.zeros_like(y) for y in ys]
    a = ([2, 0, 1], [0, 3, 7, 10], 10, 24, 8, 3)
    _, d1 = oracle.sgmv_rows(rows, x[rows], _slices(A, B, zeros, rows, 8, 24), *a)
    _, d2 = oracle.sgmv_rows(rows, 2 * x[rows], _slices(A, B, zeros, rows, 8, 24), *a)
    for j in range(3):
        assert np.array_equal(2 * d1[j], d2[j])


def test_fused_equals_per_projection():
    """Fused q/k/v (A on the rank dim, B on the output dim, block-diagonal
    product) gives bit-identical results to three separate projections."""
    spec = sy.custom_spec(dtype="bf16", n_requests=10, max_num_loras=3, max_lora_rank=16,
                          rank_choices=(4, 16))
    raw = sy.draw(spec, seed=3)
    pf = oracle.prepare_problem(raw, "qkv", fused=True)
    pp = oracle.prepare_problem(raw, "qkv", fused=False)
    rows = np.arange(pf["end"])
    uf, yf = oracle.problem_rows(pf, rows)
    up, yp = oracle.problem_rows(pp, rows)
    assert np.array_equal(uf, up)
    for a, b in zip(yf, yp):
        assert np.array_equal(a, b)
    # the fused stack really is the concatenation
    R = 16
    A0 = pf["stored"]["A"][1]
    assert np.array_equal(A0[R:2 * R], pp["stored"]["A"][1][1])
    B0 = pf["stored"]["B"][2]
    q = raw["out_dims"]["q"]
    assert np.array_equal(B0[q:q + raw["out_dims"]["k"]], pp["stored"]["B"][1][2])


def test_tiny_workload_against_einsum():
    """The tiny fp32 workload (16 routed rows) against numpy einsum in double."""
    raw = sy.draw("tiny", 0)
    for proj in ("qkv", "o"):
        p = oracle.prepare_problem(raw, proj, fused=True)
        assert p["end"] == 16
        rows = np.arange(16)
        u, ys = oracle.problem_rows(p, rows)
        x = oracle.to_f64(p["x"], "f32")
        tok_slot = np.repeat(p["lora_ids"], np.diff(p["grouped_offsets"]))
        for j, sl in enumerate(p["slices"]):
            A = sl["A"].reshape(-1)
            B = sl["B"].reshape(-1)
            R, k = p["R"], p["in_dim"]
            for t in range(16):
                s = tok_slot[t]
                a0 = sl["A_offset"] + s * sl["A_slot_stride"]
                Am = A[a0:a0 + R * k].reshape(R, k)
                b0 = sl["B_offset"] + s * sl["B_slot_stride"]
                Bm = B[b0:b0 + sl["out_dim"] * R].reshape(sl["out_dim"], R)
                uu = np.einsum("ki,i->k", Am, x[t])
                yy = oracle.to_f64(sl["y"], "f32")[t, sl["y_col0"]:sl["y_col0"] + sl["out_dim"]]
                np.testing.assert_allclose(u[t, j * R:(j + 1) * R], uu, rtol=1e-13, atol=1e-13)
                np.testing.assert_allclose(ys[j][t], yy + np.einsum("ok,k->o", Bm, uu),
                                           rtol=1e-13, atol=1e-13)


def test_generator_is_deterministic():
    a = sy.draw("decode8b", 5, with_weights=False)
    b = sy.draw("decode8b", 5, with_weights=False)
    assert np.array_equal(a["req_slot"], b["req_slot"])
    assert np.array_equal(a["x_qkv"], b["x_qkv"])
    c = sy.draw("decode8b", 6, with_weights=False)
    assert not np.array_equal(a["x_qkv"], c["x_qkv"])


def test_mlp_gate_up_fused_equals_per_projection():
    """MLP projections: gate and up fused as two slices over the same input
    give bit-identical results to two separate projections; down reads the
    intermediate activations."""
    spec = sy.custom_spec(family="mlp", intermediate=96, hidden=64, n_requests=9, max_num_loras=3,
                          rank_choices=(8, 16))
    raw = sy.draw(spec, seed=4)
    assert raw["x_gateup"].shape[1] == 64 and raw["x_down"].shape[1] == 96
    assert raw["y_gateup"].shape[1] == 192 and raw["y_down"].shape[1] == 64
    pf = oracle.prepare_problem(raw, "gateup", fused=True)
    pp = oracle.prepare_problem(raw, "gateup", fused=False)
    rows = np.arange(pf["end"])
    uf, yf = oracle.problem_rows(pf, rows)
    up, yp = oracle.problem_rows(pp, rows)
    assert np.array_equal(uf, up)
    for a, b in zip(yf, yp):
        assert np.array_equal(a, b)
    pd = oracle.prepare_problem(raw, "down")
    assert pd["in_dim"] == 96 and pd["out_dims"] == [64]


def test_token_rows_brute_force():
    """Rows of the sorted tokens of an arrival-order batch: the routed rows,
    each exactly once, grouped by slot in the order of the triple."""
    rng = np.random.default_rng(12)
    for _ in range(300):
        n = int(rng.integers(0, 12))
        slots = rng.integers(-1, 4, size=n).astype(np.int32)
        lens = rng.integers(0, 5, size=n).astype(np.int32)
        r = oracle.build_routing(slots, lens, 4)
        rows = oracle.token_rows(lens, r["perm"], r["end"])
        per_row = oracle.row_slots(slots, lens)
        assert len(rows) == r["end"] == int((per_row >= 0).sum())
        assert sorted(rows.tolist()) == np.nonzero(per_row >= 0)[0].tolist()
        for g in range(r["num_groups"]):
            seg = rows[r["grouped_offsets"][g]:r["grouped_offsets"][g + 1]]
            assert np.all(per_row[seg] == r["lora_ids"][g])


def test_per_token_definition_matches_routed_definition():
    """The per-token oracle (slot per row, no triple) and the routed oracle
    agree bit-exactly on a sorted batch; base rows come back unchanged."""
    spec = sy.custom_spec(dtype="bf16", n_requests=12, max_num_loras=4, rank_choices=(8, 16))
    raw = sy.draw(spec, seed=6)
    p = oracle.prepare_problem(raw, "qkv")
    r = p["route"]
    sorted_rows = oracle.token_rows(raw["req_len"], r["perm"], r["total_tokens"])
    # present x / y in sorted order: the routed oracle then reads rows 0..end
    ps = dict(p)
    ps["x"] = raw["x_qkv"][sorted_rows]
    ps["slices"] = [dict(sl, y=raw["y_qkv"][sorted_rows]) for sl in p["slices"]]
    rows = np.arange(r["end"])
    u1, y1 = oracle.problem_rows(ps, rows)
    slot_sorted = oracle.row_slots(raw["req_slot"], raw["req_len"])[sorted_rows]
    u2, y2 = oracle.problem_token_rows(ps, np.arange(r["total_tokens"]), slot_sorted)
    assert np.array_equal(u1, u2[:r["end"]])
    for a, b in zip(y1, y2):
        assert np.array_equal(a, b[:r["end"]])
    yin = oracle.to_f64(ps["slices"][0]["y"], "bf16")
    assert np.array_equal(y2[0][r["end"]:], yin[r["end"]:, :y2[0].shape[1]])


def test_per_token_merged_weight():
    rng = np.random.default_rng(13)
    S, R, k, o = 3, 4, 10, 6
    A = rng.standard_normal((S, R, k))
    B = rng.standard_normal((S, o, R))
    x = rng.standard_normal((7, k))
    W0 = rng.standard_normal((o, k))
    y = x @ W0.T
    slots = np.array([2, -1, 0, 0, 1, -1, 2], dtype=np.int32)
    sl = [{"A": A, "A_slot_stride": R * k, "B": B, "B_slot_stride": o * R, "out_dim": o, "y_in": y}]
    _, (yo,) = oracle.sgmv_token_slots(slots, x, sl, k, R, S)
    for t, s in enumerate(slots):
        W = W0 + (B[s] @ A[s] if s >= 0 else 0)
        np.testing.assert_allclose(yo[t], W @ x[t], rtol=1e-12, atol=1e-12)


def test_bias_merged_weight():
    """With a LoRA bias the routed rows get W0 x + b_s + B_s A_s x; the bias is
    added unscaled (vLLM page section 8, --enable-lora-bias; MAX page LoRA types)."""
    rng = np.random.default_rng(15)
    S, R, k, o = 3, 4, 9, 5
    A = rng.standard_normal((S, R, k))
    B = rng.standard_normal((S, o, R))
    bias = rng.standard_normal((S, o))
    x = rng.standard_normal((6, k))
    W0 = rng.standard_normal((o, k))
    y = x @ W0.T
    sl = [{"A": A, "A_slot_stride": R * k, "B": B, "B_slot_stride": o * R, "out_dim": o, "y_in": y,
           "bias": bias, "bias_slot_stride": o}]
    lora_ids, offs = [1, 2], [0, 2, 5]
    _, (yo,) = oracle.sgmv_rows(list(range(5)), x[:5], [dict(sl[0], y_in=y[:5])], lora_ids, offs, 5, k, R, S)
    for t in range(5):
        s_ = 1 if t < 2 else 2
        np.testing.assert_allclose(yo[t], (W0 + B[s_] @ A[s_]) @ x[t] + bias[s_], rtol=1e-12, atol=1e-12)
    _, (yt,) = oracle.sgmv_token_slots([1, 1, 2, 2, 2, -1], x, sl, k, R, S)
    np.testing.assert_allclose(yt[:5], yo, rtol=0, atol=0)
    assert np.array_equal(yt[5], y[5])


def test_openmp_build_matches_single_thread_bitwise():
    """The OpenMP build of the oracle shares the listed rows out among
    threads but computes each row exactly as the single-threaded build does:
    the results are bit-identical (routed rows and per-token rows)."""
    if not oracle.omp_available():
        pytest.skip("no OpenMP compiler here")
    spec = sy.custom_spec(max_num_loras=5, max_lora_rank=32, rank_choices=(16, 32), kind="prefill",
                          n_requests=12, len_range=(1, 40), slot_dist="uniform+base", hidden=256,
                          n_heads=8, n_kv_heads=2, head_dim=32)
    raw = sy.add_bias(sy.draw(spec, 3), 3)
    for proj in ("qkv", "o"):
        prob = oracle.prepare_problem(raw, proj)
        rows = np.arange(prob["end"], dtype=np.int32)
        u1, y1 = oracle.problem_rows(prob, rows)
        u2, y2 = oracle.problem_rows(prob, rows, parallel=True)
        assert np.array_equal(u1, u2)
        for a, b in zip(y1, y2):
            assert np.array_equal(a, b)
        slots = oracle.row_slots(raw["req_slot"], raw["req_len"])
        allr = np.arange(raw["T"], dtype=np.int32)
        _, t1 = oracle.problem_token_rows(prob, allr, slots)
        _, t2 = oracle.problem_token_rows(prob, allr, slots, parallel=True)
        for a, b in zip(t1, t2):
            assert np.array_equal(a, b)


# ------------------------------------- the delta fused into the base projection --

def test_base_rows_identity_and_selection():
    """W0 = I returns x exactly; a selection matrix (row o picks input p(o))
    returns the picked inputs exactly: no dropped, shifted or transposed
    index."""
    rng = np.random.default_rng(81)
    k = 12
    x = rng.standard_normal((5, k))
    assert np.array_equal(oracle.base_rows(np.eye(k), x), x)
    perm = rng.permutation(k)[:7]
    W = np.zeros((7, k))
    W[np.arange(7), perm] = 1.0
    assert np.array_equal(oracle.base_rows(W, x), x[:, perm])
    W2 = 2.0 * W - np.zeros_like(W)
    assert np.array_equal(oracle.base_rows(W2, x), 2.0 * x[:, perm])


def test_base_rows_matches_an_independent_product():
    """Against numpy's matrix product (another implementation) to 1e-12."""
    rng = np.random.default_rng(82)
    W = rng.standard_normal((33, 70))
    x = rng.standard_normal((9, 70))
    np.testing.assert_allclose(oracle.base_rows(W, x), x @ W.T, rtol=1e-12, atol=1e-12)


def test_fused_base_is_merged_weight():
    """The base projection with the delta fused in equals the merged-weight
    product (W0 + B_s A_s) x on routed rows and W0 x on base rows (vLLM page
    section 1), by numpy brute force on a drawn workload with base rows."""
    spec = sy.custom_spec(max_num_loras=3, max_lora_rank=16, rank_choices=(4, 16), kind="fixed",
                          fixed_slots=(2, 0, -1, 1, 0), fixed_lens=(3, 2, 4, 5, 1), hidden=32, n_heads=2,
                          n_kv_heads=1, head_dim=16)
    raw = sy.add_base_weights(sy.draw(spec, 83), 83)
    for proj in ("qkv", "o"):
        prob = oracle.prepare_problem(raw, proj)
        names = {"qkv": ["q", "k", "v"], "o": ["o"]}[proj]
        W0s = [oracle.prep_w0(raw["W0"][nm], raw["dtype"]) for nm in names]
        T = raw["T"]
        got = oracle.problem_rows_with_base(prob, np.arange(T, dtype=np.int32), W0s)
        x = oracle.to_f64(raw["x_" + proj], raw["dtype"])
        slots = np.full(T, -1)
        for g in range(len(prob["lora_ids"])):
            slots[prob["grouped_offsets"][g]:prob["grouped_offsets"][g + 1]] = prob["lora_ids"][g]
        for j, nm in enumerate(names):
            W0 = oracle.to_f64(W0s[j], raw["dtype"])
            sl = prob["slices"][j]
            R, kin = prob["R"], prob["in_dim"]
            for t in range(T):
                W = W0.copy()
                s = slots[t]
                if s >= 0:
                    Af = sl["A"].reshape(-1)[sl["A_offset"] + s * sl["A_slot_stride"]:][:R * kin].reshape(R, kin)
                    Bf = sl["B"].reshape(-1)[sl["B_offset"] + s * sl["B_slot_stride"]:][:sl["out_dim"] * R]
                    W = W + Bf.reshape(sl["out_dim"], R) @ Af
                np.testing.assert_allclose(got[j][t], W @ x[t], rtol=1e-12, atol=1e-12)
