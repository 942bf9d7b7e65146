"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.

Bars: routing bit-exact; slot preparation bit-exact; u within
1e-3 (1 + |ref|); y within 2e-2 (1 + |ref|) for bf16 and 1e-3 (1 + |ref|)
for fp32; rows at or past `end` bit-identical (NaN-payload sentinels).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import synthetic as sy

pytestmark = pytest.mark.gpu

TOL_U = 1e-3
TOL_Y = {"bf16": 2e-2, "f32": 1e-3}
SENTINEL = {"bf16": 0x7FC1, "f32": 0x7FC00001}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()


def _lk():
    import adapter_sgmv_lora_gb300 as lk
    return lk


def _dev():
    from workloads import device
    return device


def _plant_sentinels(dev, end):
    dt = dev["dtype"]
    bits = SENTINEL[dt]
    for y in dev["ys"] if dev["separate_y"] else [dev["y_all"]]:
        if y.shape[0] > end:
            if dt == "bf16":
                y[end:].view(torch.int16).fill_(bits - 0x10000 if bits > 0x7FFF else bits)
            else:
                y[end:].view(torch.int32).fill_(bits)


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _sample_rows(offs, end, rng, extra=48):
    rows = set()
    for g in range(len(offs) - 1):
        a, b = int(offs[g]), int(offs[g + 1])
        if b <= a:
            continue
        for t in (a, a + 1, b - 2, b - 1):
            if a <= t < b:
                rows.add(t)
        for base in range(a + 63, b, 64):  # around every 64-row tile boundary
            for t in (base, base + 1):
                if a <= t < b:
                    rows.add(t)
    if end > 0:
        rows.update(int(v) for v in rng.integers(0, end, size=min(extra, end)))
    return np.array(sorted(rows), dtype=np.int32)


def _poison_padding(dev, raw):
    """NaN into every A row / B column from ceil16(rank) on: with slot ranks
    passed, the kernels must never read them."""
    R = raw["max_lora_rank"]
    A, B = dev["stacks"]["A"], dev["stacks"]["B"]
    As = A if isinstance(A, list) else [A]
    Bs = B if isinstance(B, list) else [B]
    n = len(dev["names"])
    for s, r in enumerate(raw["rank"]):
        k16 = min(R, (int(r) + 15) // 16 * 16)
        if k16 >= R:
            continue
        for a in As:
            for j in range(a.shape[1] // R):
                a[s, j * R + k16:(j + 1) * R].fill_(float("nan"))
        for b in Bs:
            b[s, :, k16:].fill_(float("nan"))


# Kernel families (lora_last_call_path) each call is expected to take.
GEN = 0x1 | 0x2        # generic shrink + expand
MMA = 0x4 | 0x8        # mma.sync shrink + expand
TC = 0x10 | 0x20       # tcgen05 shrink + expand
TC_MMA = 0x10 | 0x8    # tcgen05 shrink, mma.sync expand


def run_case(raw, proj="qkv", fused=True, mode="apply", rows="all", separate_y=False, seed=0,
             slot_ranks=False, poison=False, path=None, parallel=False, host_offsets=False, host_ids=False):
    """Prepare on the device, run, compare with the oracle.  Returns the device dict.

    path: the exact OR of kernel-family bits the call(s) must have launched
    (both calls together in split mode), or None for no check.
    parallel: check with the OpenMP build of the oracle (same numbers,
    shared out over the host's cores; for full-size workloads)."""
    lk, device = _lk(), _dev()
    dev = device.prepare(raw, proj, fused=fused, separate_y=separate_y, slot_ranks=slot_ranks,
                         host_offsets=host_offsets, host_ids=host_ids)
    ref = oracle.prepare_problem(raw, proj, fused=fused)
    dt = raw["dtype"]
    # routing: library == oracle, bit-exact
    rt = dev["route_host"]
    assert np.array_equal(rt["lora_ids"], ref["route"]["lora_ids"])
    assert np.array_equal(rt["grouped_offsets"], ref["route"]["grouped_offsets"])
    assert np.array_equal(rt["perm"], ref["route"]["perm"])
    end = rt["end"]
    # stacks: lora_set_slot == oracle preparation, bit-exact
    if fused or len(dev["names"]) == 1:
        assert np.array_equal(device.torch_to_storage(dev["stacks"]["A"], dt), ref["stored"]["A"])
        assert np.array_equal(device.torch_to_storage(dev["stacks"]["B"], dt), ref["stored"]["B"])
    else:
        for j in range(len(dev["names"])):
            assert np.array_equal(device.torch_to_storage(dev["stacks"]["A"][j], dt), ref["stored"]["A"][j])
            assert np.array_equal(device.torch_to_storage(dev["stacks"]["B"][j], dt), ref["stored"]["B"][j])
    if raw.get("bias") is not None:
        got_b = dev["stacks"]["bias"]
        want_b = ref["stored"]["bias"]
        if isinstance(got_b, list):
            for gb, wb in zip(got_b, want_b):
                assert np.array_equal(device.torch_to_storage(gb, dt), wb)
        else:
            assert np.array_equal(device.torch_to_storage(got_b, dt), want_b)
    if poison:
        _poison_padding(dev, raw)
    _plant_sentinels(dev, end)
    y_before = device.y_host(dev)
    prob, routing = dev["problem"], dev["routing"]
    u = None
    if mode == "apply":
        lk.lora_sgmv_apply(prob, routing, dev["workspace"])
        taken = lk.lora_last_call_path()[0]
    else:
        nR = len(dev["names"]) * raw["max_lora_rank"]
        u = torch.full((max(end, 1), nR), float("nan"), dtype=torch.float32, device="cuda")
        lk.lora_shrink(prob, routing, u)
        taken = lk.lora_last_call_path()[0]
        lk.lora_expand(prob, routing, u)
        taken |= lk.lora_last_call_path()[0]
    torch.cuda.synchronize()
    if path is not None and end > 0:
        assert taken == path, ("kernel path", hex(taken), hex(path))
    assert lk.lora_get_device_status() == 0
    y_after = device.y_host(dev)
    # rows >= end: bit-identical (compare bit patterns: the sentinels are NaNs)
    assert np.array_equal(_bits(y_after[end:]), _bits(y_before[end:]))
    if end == 0:
        return dev
    rng = np.random.default_rng(seed)
    rr = np.arange(end, dtype=np.int32) if rows == "all" else _sample_rows(rt["grouped_offsets"], end, rng)
    u_ref, ys_ref = oracle.problem_rows(ref, rr, parallel=parallel)
    got = oracle.to_f64(y_after[rr], dt)
    col = 0
    for yj in ys_ref:
        g = got[:, col:col + yj.shape[1]]
        err = np.abs(g - yj) / (1.0 + np.abs(yj))
        assert err.max() <= TOL_Y[dt], ("y", float(err.max()), int(np.argmax(err.max(axis=1))))
        col += yj.shape[1]
    if u is not None:
        ug = u.cpu().numpy().astype(np.float64)[rr]
        err = np.abs(ug - u_ref) / (1.0 + np.abs(u_ref))
        assert err.max() <= TOL_U, ("u", float(err.max()))
    return dev


# ------------------------------------------------------------ workloads --

@pytest.mark.parametrize("proj", ["qkv", "o"])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_tiny_fp32(proj, mode):
    run_case(sy.draw("tiny", 0), proj, mode=mode, path=GEN)


@pytest.mark.parametrize("proj", ["qkv", "o"])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_decode8b_full(proj, mode):
    run_case(sy.draw("decode8b", 0), proj, mode=mode, path=MMA)


@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_many64_unfused_full(proj):
    run_case(sy.draw("many64", 0), proj, fused=False, mode="split", path=MMA)


def test_many64_separate_outputs():
    run_case(sy.draw("many64", 1), "qkv", fused=False, separate_y=True, path=MMA)


@pytest.mark.parametrize("proj", ["qkv", "o"])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_prefill8b_every_row(proj, mode):
    """Full-size ragged prefill (R = 64, 4 slots): every routed row against
    the oracle, on the tensor-core path."""
    run_case(sy.draw("prefill8b", 0), proj, mode=mode, path=TC, parallel=True)


@pytest.mark.parametrize("proj", ["qkv", "o"])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_mixed70b_every_row(proj, mode):
    """Full-size mixed 70B batch (R = 128, 16 slots, 8192 rows): every routed
    row against the oracle, on the tensor-core path."""
    run_case(sy.draw("mixed70b", 0), proj, mode=mode, path=TC, parallel=True)


@pytest.mark.parametrize("proj", ["gateup", "down"])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_mlp8b_full(proj, mode):
    """MLP projections (gate + up fused as two slices; down over the 14336-wide
    intermediate activations)."""
    run_case(sy.draw("mlp8b", 0), proj, mode=mode, path=MMA)


# -------------------------------------- checks dominated by the LoRA delta --

@pytest.mark.parametrize("mode", ["apply", "split"])
def test_delta_dominated_decode(mode):
    """y_in = 0 and B scaled so the delta is of order one or more: the
    2e-2 (1 + |ref|) bar then measures the delta itself (decode shapes,
    mma.sync path)."""
    raw = sy.emphasize_delta(sy.draw("decode8b", 31), 40.0)
    run_case(raw, "qkv", mode=mode, path=MMA)
    run_case(raw, "o", mode=mode, path=MMA)


@pytest.mark.parametrize("R", [16, 64, 128])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_delta_dominated_long_groups(R, mode):
    """As above on the tensor-core path for long groups (ragged 128-row
    tiles), ranks 16, 64 and 128."""
    spec = _spec(max_num_loras=5, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(4, 3, 2, 1, 0, -1), fixed_lens=(130, 255, 128, 300, 97, 7),
                 hidden=512, n_heads=8, n_kv_heads=2, head_dim=64)
    raw = sy.emphasize_delta(sy.draw(spec, 32 + R), 40.0)
    run_case(raw, "qkv", mode=mode, path=TC if R >= 64 else TC_MMA)
    run_case(raw, "o", mode=mode, path=TC if R >= 64 else TC_MMA)


def test_delta_dominated_fp32_and_bias():
    """fp32 generic kernels, and the general mma.sync kernels with a bias and
    true ranks, with y_in = 0 and an order-one delta."""
    spec = _spec(dtype="f32", max_lora_rank=32, rank_choices=(8, 32), n_requests=25)
    run_case(sy.emphasize_delta(sy.draw(spec, 41), 40.0), "qkv", mode="split", path=GEN)
    raw = sy.add_bias(sy.emphasize_delta(sy.draw("decode8b", 42), 40.0), 42, scale=1.0)
    run_case(raw, "qkv", mode="apply", slot_ranks=True, poison=True, path=MMA)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_mlp_long_groups_tensor_core_path(mode):
    spec = _spec(family="mlp", hidden=512, intermediate=1024, max_num_loras=3, max_lora_rank=64,
                 rank_choices=(32, 64), kind="fixed", fixed_slots=(2, 0, 1, -1),
                 fixed_lens=(300, 513, 200, 11))
    run_case(sy.draw(spec, 9), "gateup", mode=mode, path=TC)
    run_case(sy.draw(spec, 10), "down", mode=mode, path=TC)


def run_unsorted(raw, proj="qkv", mode="apply", path=None, parallel=False, host_ids=False):
    """x and y rows in ARRIVAL order; token_rows maps the sorted order to rows.
    Compared with the per-token oracle (slot of each row, no routing triple).
    path: the exact kernel families the call(s) must take (None: no check).
    host_ids: the routing carries host copies of the offsets and slot ids."""
    lk, device = _lk(), _dev()
    dev = device.prepare(raw, proj)
    rt = dev["route_host"]
    rows = lk.lora_build_token_rows(raw["req_len"], rt["perm"], rt["end"])
    assert np.array_equal(rows, oracle.token_rows(raw["req_len"], rt["perm"], rt["end"]))
    tr = torch.from_numpy(rows).cuda() if rt["end"] > 0 else None
    routing = lk.Routing(dev["routing"].lora_ids, dev["routing"].grouped_offsets, rt["num_groups"], rt["end"], tr)
    if host_ids:
        routing.host_grouped_offsets = np.asarray(rt["grouped_offsets"], dtype=np.int32)
        routing.host_lora_ids = np.asarray(rt["lora_ids"], dtype=np.int32)[: rt["num_groups"]]
    y_before = device.y_host(dev)
    if mode == "apply":
        lk.lora_sgmv_apply(dev["problem"], routing, dev["workspace"])
        taken = lk.lora_last_call_path()[0]
    else:
        nR = len(dev["names"]) * raw["max_lora_rank"]
        u = torch.empty((max(rt["end"], 1), nR), dtype=torch.float32, device="cuda")
        lk.lora_shrink(dev["problem"], routing, u)
        taken = lk.lora_last_call_path()[0]
        lk.lora_expand(dev["problem"], routing, u)
        taken |= lk.lora_last_call_path()[0]
    torch.cuda.synchronize()
    assert lk.lora_get_device_status() == 0
    if path is not None:
        assert taken == path, ("kernel path", hex(taken), hex(path))
    y_after = device.y_host(dev)
    ref = oracle.prepare_problem(raw, proj)
    slots = oracle.row_slots(raw["req_slot"], raw["req_len"])
    all_rows = np.arange(raw["T"], dtype=np.int32)
    _, ys = oracle.problem_token_rows(ref, all_rows, slots, parallel=parallel)
    got = oracle.to_f64(y_after, raw["dtype"])
    base = slots < 0
    assert np.array_equal(_bits(y_after[base]), _bits(y_before[base]))
    col = 0
    for yj in ys:
        g = got[:, col:col + yj.shape[1]]
        err = (np.abs(g - yj) / (1.0 + np.abs(yj)))[~base]
        assert err.max() <= TOL_Y[raw["dtype"]], float(err.max())
        col += yj.shape[1]


@pytest.mark.parametrize("mode", ["apply", "split"])
@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_unsorted_decode_batch_token_rows(mode, proj):
    run_unsorted(sy.draw("decode8b", 3), proj, mode)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_unsorted_multi_token_requests(mode):
    spec = _spec(max_num_loras=5, max_lora_rank=32, rank_choices=(16, 32), kind="prefill", n_requests=14,
                 len_range=(1, 150), slot_dist="uniform+base", hidden=1024, n_heads=16, n_kv_heads=4,
                 head_dim=64)
    run_unsorted(sy.draw(spec, 11), "qkv", mode)
    run_unsorted(sy.draw(_spec(dtype="f32", n_requests=20), 12), "qkv", mode)


@pytest.mark.parametrize("mode", ["apply", "split"])
@pytest.mark.parametrize("R", [16, 64, 128])
def test_unsorted_long_groups_tensor_core(mode, R):
    """Unsorted (arrival-order) batches of long groups on the tcgen05 path:
    the shrink gathers x rows through token_rows (16-byte async copies into
    the swizzled stages), the expand reads and writes its scattered y rows
    itself.  Ragged 128-row tiles; per-token oracle on every row."""
    spec = _spec(max_num_loras=5, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(2, -1, 0, 4, 1, 3, 0, 2), fixed_lens=(130, 17, 255, 128, 97, 300, 64, 90),
                 hidden=512, n_heads=8, n_kv_heads=2, head_dim=64)
    want = TC if R >= 64 else TC_MMA
    run_unsorted(sy.draw(spec, 110 + R), "qkv", mode, path=want)
    run_unsorted(sy.draw(spec, 111 + R), "o", mode, path=want)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_unsorted_prefill8b_tensor_core(mode):
    """The full-size prefill batch in arrival order (token_rows), on tcgen05,
    every row against the per-token oracle."""
    run_unsorted(sy.draw("prefill8b", 7), "qkv", mode, path=TC, parallel=True)


def test_unsorted_long_groups_bad_row_is_flagged():
    """An out-of-range token_rows entry on the tcgen05 path raises
    LORA_DEV_BAD_ROW (the tile holding it is skipped)."""
    lk, device = _lk(), _dev()
    spec = _spec(max_num_loras=3, max_lora_rank=64, rank_choices=(64,), kind="fixed",
                 fixed_slots=(1, 0, 2), fixed_lens=(200, 300, 150), hidden=256, n_heads=4, n_kv_heads=2,
                 head_dim=64)
    raw = sy.draw(spec, 120)
    dev = device.prepare(raw, "qkv")
    rt = dev["route_host"]
    rows = lk.lora_build_token_rows(raw["req_len"], rt["perm"], rt["end"])
    rows[5] = raw["T"] + 7
    routing = lk.Routing(dev["routing"].lora_ids, dev["routing"].grouped_offsets, rt["num_groups"], rt["end"],
                         torch.from_numpy(rows).cuda())
    assert lk.lora_get_device_status() == 0
    lk.lora_sgmv_apply(dev["problem"], routing, dev["workspace"])
    assert lk.lora_last_call_path()[0] == TC
    assert lk.lora_get_device_status() & lk.DEV_BAD_ROW


def test_token_rows_out_of_range_is_flagged_and_skipped():
    lk, device = _lk(), _dev()
    raw = sy.draw("decode8b", 4)
    dev = device.prepare(raw, "qkv")
    rt = dev["route_host"]
    rows = lk.lora_build_token_rows(raw["req_len"], rt["perm"], rt["end"])
    rows[3] = raw["T"] + 100
    routing = lk.Routing(dev["routing"].lora_ids, dev["routing"].grouped_offsets, rt["num_groups"], rt["end"],
                         torch.from_numpy(rows).cuda())
    assert lk.lora_get_device_status() == 0
    lk.lora_sgmv_apply(dev["problem"], routing, dev["workspace"])
    assert lk.lora_get_device_status() & lk.DEV_BAD_ROW


# ------------------------------------------ LoRA bias and true-rank hints --

@pytest.mark.parametrize("mode", ["apply", "split"])
def test_bias_decode(mode):
    run_case(sy.add_bias(sy.draw("decode8b", 5), 5), "qkv", mode=mode)
    run_case(sy.add_bias(sy.draw("decode8b", 6), 6), "o", mode=mode)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_bias_and_ranks_long_groups(mode):
    """tcgen05 path with bias and rank hints (ranks 16/32/64 of max 64), NaN in
    the padding the hints skip."""
    spec = _spec(max_num_loras=4, max_lora_rank=64, rank_choices=(16, 32, 64), kind="fixed",
                 fixed_slots=(3, 0, 2, 1, -1), fixed_lens=(150, 300, 129, 260, 9), hidden=512, n_heads=8,
                 n_kv_heads=2, head_dim=64)
    for seed in (1, 2):
        raw = sy.add_bias(sy.draw(spec, seed), seed)
        run_case(raw, "qkv", mode=mode, slot_ranks=True, poison=True, path=TC)
        run_case(raw, "o", mode=mode, slot_ranks=True, poison=True, path=TC)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_rank_hints_short_groups(mode):
    """mma.sync path with rank hints (ranks 16..128 of max 128), NaN padding."""
    spec = _spec(max_num_loras=6, max_lora_rank=128, rank_choices=(16, 48, 64, 128), n_requests=40,
                 hidden=512, n_heads=8, n_kv_heads=2, head_dim=64)
    raw = sy.add_bias(sy.draw(spec, 3), 3)
    run_case(raw, "qkv", mode=mode, slot_ranks=True, poison=True)
    run_case(sy.draw(spec, 4), "o", mode=mode, slot_ranks=True, poison=True)


def test_bias_and_ranks_generic_path():
    spec = _spec(dtype="f32", max_lora_rank=32, rank_choices=(8, 32), n_requests=25)
    run_case(sy.add_bias(sy.draw(spec, 1), 1), "qkv", mode="split", slot_ranks=True, poison=True)


def test_bias_unsorted_batch():
    run_unsorted(sy.add_bias(sy.draw("decode8b", 7), 7), "qkv", "apply")


# ------------------------------------------------------------ edge cases --

def _spec(**kw):
    return sy.custom_spec(**kw)


@pytest.mark.parametrize("R", [16, 32, 64, 128])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_rank_variants_ragged_tiles(R, mode):
    """Group lengths straddling 64-row tiles: 1, 63, 64, 65, 127, 130, 200."""
    spec = _spec(max_num_loras=7, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(0, 1, 2, 3, 4, 5, 6, -1), fixed_lens=(1, 63, 64, 65, 127, 130, 200, 9),
                 hidden=256, n_heads=8, n_kv_heads=2, head_dim=32)
    run_case(sy.draw(spec, 3), "qkv", mode=mode, path=MMA)
    run_case(sy.draw(spec, 4), "o", mode=mode, path=MMA)
    if mode == "apply" and R >= 64:  # the routing's host offsets: long groups on tcgen05
        run_case(sy.draw(spec, 3), "qkv", mode=mode, path=0x10 | 0x20 | 0x4 | 0x8, host_offsets=True)


@pytest.mark.parametrize("mode", ["apply", "split"])
@pytest.mark.parametrize("ranks", [False, True])
def test_short_groups_wide_expand_tiles(mode, ranks):
    """Groups of at most 32 rows on average take the expand's 32-row tiles,
    here 256 columns wide (a small grid): lengths 1, 31, 32, 33, 40, 3, 8 and
    0 (tiles of 32 with ragged ends), slices narrower than one block; also
    with the true ranks passed (the general kernels)."""
    spec = _spec(max_num_loras=8, max_lora_rank=16, rank_choices=(8, 16), kind="fixed",
                 fixed_slots=(7, 6, 5, 4, 3, 2, 1, 0, -1), fixed_lens=(1, 31, 32, 33, 40, 3, 8, 0, 6),
                 hidden=1024, n_heads=16, n_kv_heads=4, head_dim=64)
    run_case(sy.draw(spec, 11), "qkv", mode=mode, slot_ranks=ranks, poison=ranks)
    run_case(sy.draw(spec, 12), "o", mode=mode, slot_ranks=ranks, poison=ranks)


@pytest.mark.parametrize("mode", ["apply", "split"])
@pytest.mark.parametrize("ranks", [False, True])
def test_short_groups_wide_outputs(mode, ranks):
    """Short groups with outputs wide enough (gate + up of 2 x 8192 columns)
    that 32-row x 512-column expand tiles already give two CTAs per SM; the
    down projection (1024 columns) takes the 256-column tiles.  Same ragged
    lengths as above; plain and general kernels."""
    spec = _spec(family="mlp", intermediate=8192, max_num_loras=8, max_lora_rank=16, rank_choices=(8, 16),
                 kind="fixed", fixed_slots=(7, 6, 5, 4, 3, 2, 1, 0, -1), fixed_lens=(1, 31, 32, 33, 40, 3, 8, 0, 6),
                 hidden=1024)
    run_case(sy.draw(spec, 13), "gateup", mode=mode, slot_ranks=ranks, poison=ranks)
    run_case(sy.draw(spec, 14), "down", mode=mode, slot_ranks=ranks, poison=ranks)


@pytest.mark.parametrize("mode", ["apply", "split"])
def test_short_groups_many_adapters_wide_outputs(mode):
    """40 adapters, 300 one-token requests, gate + up of 2 x 4096 columns: a
    grid of several waves of 32 x 512 expand tiles over many small groups,
    checked on every routed row."""
    spec = _spec(family="mlp", intermediate=4096, hidden=512, max_num_loras=40, max_lora_rank=16,
                 rank_choices=(8, 16), n_requests=300, base_prob=0.1)
    for seed in (21, 22):
        run_case(sy.draw(spec, seed), "gateup", mode=mode)


@pytest.mark.parametrize("R", [16, 32])
def test_apply_split_planes_ragged_groups(R):
    """The apply's shrink splits K into partial planes for small batches;
    groups of 1, 31, 32, 33, 64, 70 and 100 rows, input width 1024."""
    spec = _spec(max_num_loras=7, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(6, 5, 4, 3, 2, 1, 0, -1), fixed_lens=(1, 31, 32, 33, 64, 70, 100, 5),
                 hidden=1024, n_heads=16, n_kv_heads=4, head_dim=64)
    run_case(sy.draw(spec, 5), "qkv", mode="apply", path=MMA)
    run_case(sy.draw(spec, 6), "o", mode="apply", path=MMA)


@pytest.mark.parametrize("R", [16, 32, 64, 128])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_long_groups_tensor_core_shrink(R, mode):
    """Long groups (the tcgen05 shrink): 128-row tiles with ragged ends,
    lengths 100, 127, 128, 129, 300 and 1000."""
    spec = _spec(max_num_loras=6, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(5, 4, 3, 2, 1, 0, -1), fixed_lens=(100, 127, 128, 129, 300, 1000, 7),
                 hidden=256, n_heads=8, n_kv_heads=2, head_dim=32)
    want = TC if R >= 64 else TC_MMA
    run_case(sy.draw(spec, 7), "qkv", mode=mode, path=want)
    run_case(sy.draw(spec, 8), "o", mode=mode, path=want)


@pytest.mark.parametrize("groups", [128, 132])
@pytest.mark.parametrize("mode", ["apply", "split"])
def test_many_long_groups(groups, mode):
    """128 long groups fill the persistent tcgen05 expand's cached routing
    exactly; 132 exceed it (the apply then pairs the tcgen05 shrink with the
    mma.sync expand).  100 rows per group, rank 64."""
    spec = _spec(max_num_loras=groups, max_lora_rank=64, rank_choices=(32, 64), kind="fixed",
                 fixed_slots=tuple(range(groups - 1, -1, -1)) + (-1,), fixed_lens=(100,) * groups + (5,),
                 hidden=128, n_heads=4, n_kv_heads=4, head_dim=32)
    run_case(sy.draw(spec, 21), "qkv", mode=mode, path=TC if groups <= 128 else TC_MMA)


def test_wait_timeout_is_reported_and_context_survives():
    """A bounded wait that runs out (a barrier nothing completes) sets
    LORA_DEV_TIMEOUT, no fault; afterwards the context still computes."""
    lk = _lk()
    assert lk.lora_get_device_status() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    lk.lora_selftest_wait_timeout(1 << 12)
    t1.record()
    torch.cuda.synchronize()
    assert lk.lora_get_device_status() == 8  # LORA_DEV_TIMEOUT, read and cleared
    assert lk.lora_get_device_status() == 0
    assert t0.elapsed_time(t1) < 5000.0
    run_case(sy.draw("tiny", 0), "qkv")


def test_all_base_is_noop():
    spec = _spec(kind="fixed", fixed_slots=(-1, -1), fixed_lens=(3, 4))
    dev = run_case(sy.draw(spec, 0), "qkv")
    assert dev["route_host"]["end"] == 0


def test_zero_length_groups_and_unsorted_arrivals():
    spec = _spec(max_num_loras=5, kind="fixed", fixed_slots=(3, -1, 0, 4, 0, 2, 1, -1),
                 fixed_lens=(5, 2, 0, 0, 7, 66, 0, 3), hidden=128)
    run_case(sy.draw(spec, 0), "qkv", mode="split")


def test_unaligned_shapes_take_generic_path():
    """in_dim not a multiple of 64 and outputs not multiples of 8: generic kernels."""
    spec = _spec(hidden=72, n_heads=3, n_kv_heads=1, head_dim=12, max_lora_rank=16, n_requests=40)
    run_case(sy.draw(spec, 0), "qkv", mode="split")
    run_case(sy.draw(spec, 1), "qkv", mode="apply")


def test_rank_not_in_fast_set():
    spec = _spec(max_lora_rank=8, rank_choices=(4, 8), n_requests=30)
    run_case(sy.draw(spec, 0), "qkv", mode="split")


def test_fp32_larger():
    spec = _spec(dtype="f32", hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, max_lora_rank=32,
                 rank_choices=(16, 32), kind="prefill", n_requests=6, len_range=(1, 150),
                 slot_dist="uniform+base")
    run_case(sy.draw(spec, 0), "qkv", mode="split")


def test_deterministic():
    lk, device = _lk(), _dev()
    raw = sy.draw("decode8b", 2)
    outs = []
    for _ in range(2):
        dev = device.prepare(raw, "qkv")
        lk.lora_sgmv_apply(dev["problem"], dev["routing"], dev["workspace"])
        torch.cuda.synchronize()
        outs.append(device.y_host(dev))
    assert np.array_equal(outs[0], outs[1])


def test_pages_base_only_fallback_leaves_y_unchanged():
    """The MAX page's base-only fallback: an all-zero adapter in slot 0 with
    every token routed to it is a no-op in value."""
    lk, device = _lk(), _dev()
    spec = _spec(max_num_loras=2, kind="fixed", fixed_slots=(0,), fixed_lens=(50,), rank_choices=(16,))
    raw = sy.draw(spec, 0)
    for p in sy.PROJS:
        raw["B"][p][0] = np.zeros_like(raw["B"][p][0])
    dev = device.prepare(raw, "qkv")
    before = device.y_host(dev)
    lk.lora_sgmv_apply(dev["problem"], dev["routing"], dev["workspace"])
    torch.cuda.synchronize()
    after = device.y_host(dev)
    a = oracle.to_f64(before, "bf16")
    b = oracle.to_f64(after, "bf16")
    assert np.array_equal(a, b)  # equal in value (+0 / -0 allowed)


@pytest.mark.parametrize("bad", ["slot", "offsets", "end"])
def test_invalid_device_routing_is_flagged_and_skipped(bad):
    lk, device = _lk(), _dev()
    raw = sy.draw("decode8b", 0)
    dev = device.prepare(raw, "qkv")
    rt = dev["route_host"]
    ids = rt["lora_ids"].copy()
    offs = rt["grouped_offsets"].copy()
    if bad == "slot":
        ids[1] = raw["max_num_loras"] + 3
        flag = lk.DEV_BAD_SLOT
    elif bad == "offsets":
        offs[2], offs[3] = offs[3], offs[2]
        flag = lk.DEV_BAD_OFFSETS
    else:
        offs[-1] -= 1
        flag = lk.DEV_BAD_END
    routing = lk.Routing(torch.from_numpy(ids).cuda(), torch.from_numpy(offs).cuda(), rt["num_groups"],
                         rt["end"])
    assert lk.lora_get_device_status() == 0
    before = device.y_host(dev)
    lk.lora_sgmv_apply(dev["problem"], routing, dev["workspace"])
    assert lk.lora_get_device_status() & flag
    assert np.array_equal(_bits(device.y_host(dev)), _bits(before))
    assert lk.lora_get_device_status() == 0  # read-and-clear


# ------------------------- the triple's host copy as launch parameters --

@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_decode8b_host_triple(proj):
    """With host copies of the offsets and the slot ids the mma.sync shrink
    locates its tiles from its launch parameters; same results."""
    run_case(sy.draw("decode8b", 5), proj, mode="apply", path=MMA, host_ids=True)


def test_host_triple_64_groups_unfused_ranks_bias():
    """64 groups (the most a launch carries), per-projection stacks; and a
    bias with true ranks (general kernels)."""
    run_case(sy.draw("many64", 6), "qkv", fused=False, mode="apply", path=MMA, host_ids=True)
    raw = sy.add_bias(sy.emphasize_delta(sy.draw("decode8b", 43), 40.0), 43, scale=1.0)
    run_case(raw, "qkv", mode="apply", slot_ranks=True, poison=True, path=MMA, host_ids=True)


def test_host_triple_unsorted_and_per_group():
    run_unsorted(sy.draw("decode8b", 7), "qkv", "apply", path=MMA, host_ids=True)
    run_case(sy.draw("mixed64", 2), "o", mode="apply", path=SPLIT, parallel=True, host_ids=True)


def test_host_triple_beyond_the_tile_table():
    """More 64-row tiles than a launch's tile table holds (100 groups of 90
    rows: 200 tiles): the shrink locates its tiles in the device triple
    instead; same results."""
    spec = _spec(max_num_loras=100, max_lora_rank=16, rank_choices=(16,), kind="fixed",
                 fixed_slots=tuple(range(99, -1, -1)) + (-1,), fixed_lens=(90,) * 100 + (3,),
                 hidden=256, n_heads=8, n_kv_heads=2, head_dim=32)
    run_case(sy.draw(spec, 44), "qkv", mode="apply", path=MMA, host_ids=True)
    run_case(sy.draw(spec, 45), "o", mode="apply", path=MMA, host_ids=True)


@pytest.mark.parametrize("what", ["ids", "offsets"])
def test_device_triple_differing_from_host_copy_is_flagged(what):
    """The shrink works from the host copy; the expand compares the device
    triple with it, and on a difference flags LORA_DEV_BAD_OFFSETS and skips
    its work: y keeps its old contents."""
    lk, device = _lk(), _dev()
    raw = sy.draw("decode8b", 8)
    dev = device.prepare(raw, "qkv", host_ids=True)
    rt = dev["route_host"]
    r = dev["routing"]
    ids = np.asarray(rt["lora_ids"], dtype=np.int32).copy()
    offs = np.asarray(rt["grouped_offsets"], dtype=np.int32).copy()
    if what == "ids":
        ids[0] = (ids[0] + 1) % raw["max_num_loras"]          # still a valid slot
    else:
        assert offs[2] > offs[1] + 1
        offs[1] += 1                                          # still a valid triple
    assert not (np.array_equal(ids, rt["lora_ids"]) and np.array_equal(offs, rt["grouped_offsets"]))
    bad = lk.Routing(torch.from_numpy(ids).cuda(), torch.from_numpy(offs).cuda(), r.num_groups, r.end,
                     None, r.host_grouped_offsets, r.host_lora_ids)
    assert lk.lora_get_device_status() == 0
    before = device.y_host(dev)
    lk.lora_sgmv_apply(dev["problem"], bad, dev["workspace"])
    assert lk.lora_last_call_path()[0] == MMA
    assert lk.lora_get_device_status() & lk.DEV_BAD_OFFSETS
    assert np.array_equal(_bits(device.y_host(dev)), _bits(before))


def test_workspace_too_small_is_rejected():
    lk, device = _lk(), _dev()
    dev = device.prepare(sy.draw("decode8b", 0), "o")
    with pytest.raises(lk.LoraError) as e:
        lk.lora_sgmv_apply(dev["problem"], dev["routing"], dev["workspace"][:10])
    assert e.value.status == 8


# --------------------------------------- the delta fused into the base GEMM --

BASE = 0x100


def run_base_case(raw, proj="qkv", rows="all", slot_ranks=False, poison=False, path=None, parallel=True,
                  seed=0):
    """lora_base_gemm_apply against the oracle's fused definition: every row
    (routed rows: W0 x + delta; base rows: W0 x), one rounding."""
    lk, device = _lk(), _dev()
    dev = device.prepare(raw, proj, slot_ranks=slot_ranks)
    if poison:
        _poison_padding(dev, raw)
    names = dev["names"]
    dt = raw["dtype"]
    W0s = [oracle.prep_w0(raw["W0"][nm], dt) for nm in names]
    W0d = [device.storage_to_torch(w, dt) for w in W0s]
    dev["y_all"].fill_(float("nan"))  # y is written, never read
    lk.lora_base_gemm_apply(dev["problem"], dev["routing"], W0d, dev["workspace"])
    bits, _ = lk.lora_last_call_path()
    torch.cuda.synchronize()
    assert lk.lora_get_device_status() == 0
    if path is not None:
        assert bits == path, hex(bits)
    ref = oracle.prepare_problem(raw, proj)
    T = raw["T"]
    if rows == "all":
        rr = np.arange(T, dtype=np.int32)
    else:
        rr = np.unique(np.concatenate([_sample_rows(ref["grouped_offsets"], ref["end"], np.random.default_rng(seed)),
                                       np.arange(ref["end"], T, max(1, (T - ref["end"]) // 40), dtype=np.int32),
                                       np.array([T - 1], dtype=np.int32)])).astype(np.int32)
    ys = oracle.problem_rows_with_base(ref, rr, W0s, parallel=parallel)
    got = oracle.to_f64(device.y_host(dev)[rr], dt)
    col = 0
    for yj in ys:
        g = got[:, col:col + yj.shape[1]]
        err = np.abs(g - yj) / (1.0 + np.abs(yj))
        assert err.max() <= TOL_Y[dt], ("y", float(err.max()))
        col += yj.shape[1]
    return dev


@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_base_gemm_decode8b_every_row(proj):
    """Decode batch at full size (256 rows, 8 slots, base rows included)."""
    raw = sy.add_base_weights(sy.draw("decode8b", 90), 90)
    run_base_case(raw, proj, path=BASE | 0x4)


@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_base_gemm_prefill8b_sampled(proj):
    """Ragged prefill at full size (R = 64): group edges, 64-row boundaries,
    random routed rows and a spread of base rows."""
    raw = sy.add_base_weights(sy.draw("prefill8b", 91), 91)
    run_base_case(raw, proj, rows="sample", path=BASE | 0x10)


@pytest.mark.parametrize("R", [16, 32, 64, 128])
def test_base_gemm_ragged_tiles(R):
    """Groups straddling the 128-row tiles (several groups per tile), a
    partial last tile, slices narrower than a column block."""
    spec = _spec(max_num_loras=7, max_lora_rank=R, rank_choices=(R // 2, R), kind="fixed",
                 fixed_slots=(0, 1, 2, 3, 4, 5, 6, -1), fixed_lens=(1, 63, 64, 65, 127, 130, 200, 9),
                 hidden=256, n_heads=8, n_kv_heads=2, head_dim=32)
    raw = sy.add_base_weights(sy.draw(spec, 92 + R), 92 + R)
    run_base_case(raw, "qkv")
    run_base_case(raw, "o")


def test_base_gemm_bias_ranks_and_delta_dominated():
    """Bias and true ranks (NaN past them) with a delta of order one."""
    spec = _spec(max_num_loras=4, max_lora_rank=64, rank_choices=(16, 32, 64), kind="fixed",
                 fixed_slots=(3, 0, 2, 1, -1), fixed_lens=(150, 300, 29, 260, 9), hidden=512, n_heads=8,
                 n_kv_heads=2, head_dim=64)
    raw = sy.add_base_weights(sy.add_bias(sy.emphasize_delta(sy.draw(spec, 96), 40.0), 96, scale=1.0), 96)
    run_base_case(raw, "qkv", slot_ranks=True, poison=True, path=BASE | 0x10)
    run_base_case(raw, "o", slot_ranks=True, poison=True)


def test_base_gemm_decode_shapes():
    """Decode-sized batches: bias, true ranks with NaN past them and an
    order-one delta; rank 32 with a row count that is not a multiple of 16;
    a single row; a two-stage input; a batch of base rows only."""
    spec = _spec(max_num_loras=6, max_lora_rank=16, rank_choices=(8, 16), kind="decode", n_requests=200,
                 base_prob=0.2, slot_dist="uniform", hidden=512, n_heads=8, n_kv_heads=4, head_dim=64)
    raw = sy.add_base_weights(sy.add_bias(sy.emphasize_delta(sy.draw(spec, 99), 40.0), 99, scale=1.0), 99)
    run_base_case(raw, "qkv", slot_ranks=True, poison=True, path=BASE | 0x4)
    run_base_case(raw, "o", slot_ranks=True, poison=True, path=BASE | 0x4)
    spec = _spec(max_num_loras=3, max_lora_rank=32, rank_choices=(32,), kind="fixed", fixed_slots=(2, 0, 1, -1),
                 fixed_lens=(9, 17, 5, 6), hidden=256, n_heads=4, n_kv_heads=4, head_dim=64)
    run_base_case(sy.add_base_weights(sy.draw(spec, 100), 100), "qkv", path=BASE | 0x4)
    spec = _spec(max_num_loras=2, max_lora_rank=16, rank_choices=(16,), kind="fixed", fixed_slots=(1,),
                 fixed_lens=(1,), hidden=256, n_heads=4, n_kv_heads=4, head_dim=64)
    run_base_case(sy.add_base_weights(sy.draw(spec, 101), 101), "o", path=BASE | 0x4)
    spec = _spec(max_num_loras=2, max_lora_rank=16, rank_choices=(16,), kind="fixed", fixed_slots=(0, 1, -1),
                 fixed_lens=(30, 40, 20), hidden=128, n_heads=2, n_kv_heads=2, head_dim=128)
    run_base_case(sy.add_base_weights(sy.draw(spec, 102), 102), "qkv", path=BASE | 0x4)
    spec = _spec(kind="fixed", fixed_slots=(-1, -1), fixed_lens=(70, 90), hidden=256, n_heads=4, n_kv_heads=4,
                 head_dim=64)
    run_base_case(sy.add_base_weights(sy.draw(spec, 103), 103), "qkv", path=BASE)


def test_base_gemm_all_base_rows_and_fp32():
    """No routed rows (the base projection alone), and the generic kernel for fp32."""
    spec = _spec(kind="fixed", fixed_slots=(-1, -1), fixed_lens=(70, 90), hidden=256, n_heads=8, n_kv_heads=2,
                 head_dim=32)
    raw = sy.add_base_weights(sy.draw(spec, 97), 97)
    run_base_case(raw, "qkv", path=BASE)
    spec = _spec(dtype="f32", max_lora_rank=32, rank_choices=(8, 32), n_requests=25)
    raw = sy.add_base_weights(sy.draw(spec, 98), 98)
    run_base_case(raw, "qkv", path=BASE | 0x1)


# --------------------------------------------- kernels picked per group --

SPLIT = 0x10 | 0x20 | 0x4 | 0x8   # tcgen05 shrink + expand for long groups, mma.sync for short ones


@pytest.mark.parametrize("proj", ["qkv", "o"])
def test_mixed64_kernels_per_group_every_row(proj):
    """A few long prefill groups among many one-token groups, with the host
    copy of the offsets: the long groups run on tcgen05 and the short ones on
    mma.sync in the same call; every routed row against the oracle."""
    run_case(sy.draw("mixed64", 0), proj, mode="apply", path=SPLIT, parallel=True, host_offsets=True)


def test_mixed64_without_host_offsets_takes_one_path():
    """Without the host copy the call picks one path from the average group
    length (here mma.sync for everything); same results."""
    lk, device = _lk(), _dev()
    raw = sy.draw("mixed64", 1)
    dev = device.prepare(raw, "qkv", host_offsets=True)
    r = dev["routing"]
    plain = lk.Routing(r.lora_ids, r.grouped_offsets, r.num_groups, r.end)
    lk.lora_sgmv_apply(dev["problem"], plain, dev["workspace"])
    assert lk.lora_last_call_path()[0] == MMA
    torch.cuda.synchronize()
    assert lk.lora_get_device_status() == 0
    ref = oracle.prepare_problem(raw, "qkv")
    end = ref["end"]
    _, ys = oracle.problem_rows(ref, np.arange(end, dtype=np.int32), parallel=True)
    got = oracle.to_f64(device.y_host(dev), "bf16")
    col = 0
    for yj in ys:
        err = np.abs(got[:end, col:col + yj.shape[1]] - yj) / (1.0 + np.abs(yj))
        assert err.max() <= TOL_Y["bf16"], float(err.max())
        col += yj.shape[1]


@pytest.mark.parametrize("R", [64, 128])
def test_kernels_per_group_ragged_and_ranks(R):
    """Long groups of 64 (the threshold), 65, 129 and 300 rows among groups of
    1 to 63 rows, with and without true ranks (NaN past them) and a bias."""
    spec = _spec(max_num_loras=10, max_lora_rank=R, rank_choices=(16, R), kind="fixed",
                 fixed_slots=(9, 8, 7, 6, 5, 4, 3, 2, 1, 0, -1), fixed_lens=(1, 64, 2, 65, 63, 129, 17, 300, 5, 33, 8),
                 hidden=512, n_heads=8, n_kv_heads=2, head_dim=64)
    run_case(sy.draw(spec, 100 + R), "qkv", mode="apply", path=SPLIT, host_offsets=True)
    run_case(sy.draw(spec, 101 + R), "o", mode="apply", path=SPLIT, host_offsets=True)
    raw = sy.add_bias(sy.draw(spec, 102 + R), 102 + R)
    run_case(raw, "qkv", mode="apply", slot_ranks=True, poison=True, path=SPLIT, host_offsets=True)


# ------------------------------------- tensor-core apply: grid extremes --

@pytest.mark.parametrize("host_offsets", [False, True])
def test_tc_apply_few_tiles_long_input(host_offsets):
    """Eight 128-row tiles (four groups of 200 rows) with in = 4096: the
    apply's shrink splits K over 4-CTA clusters (n*R = 384 and 128), the
    partials exchanged through distributed shared memory.  Every row against
    the oracle with an order-one delta, with and without the routing's host
    copy."""
    spec = _spec(max_num_loras=4, max_lora_rank=128, rank_choices=(64, 128), kind="fixed",
                 fixed_slots=(3, 0, 2, 1, -1), fixed_lens=(200, 200, 200, 200, 11),
                 hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128)
    raw = sy.emphasize_delta(sy.draw(spec, 51), 40.0)
    run_case(raw, "qkv", mode="apply", path=TC, parallel=True, host_offsets=host_offsets)
    run_case(raw, "o", mode="apply", path=TC, parallel=True, host_offsets=host_offsets)


def test_tc_apply_many_tiles_short_input():
    """448 tiles (eight groups of 7100 rows) with in = 128: one shrink CTA
    per tile over several waves, and the persistent expand's units spread
    over every SM.  Ranks 64, every row against the oracle."""
    spec = _spec(max_num_loras=8, max_lora_rank=64, rank_choices=(32, 64), kind="fixed",
                 fixed_slots=tuple(range(8)) + (-1,), fixed_lens=(7100,) * 8 + (5,),
                 hidden=128, n_heads=4, n_kv_heads=2, head_dim=32)
    raw = sy.draw(spec, 52)
    run_case(raw, "qkv", mode="apply", path=TC, parallel=True)
    run_case(raw, "o", mode="apply", path=TC, parallel=True)


def test_tc_apply_deterministic():
    """The K-split shrink sums its CTAs' partials in rank order: repeated
    applies give bit-identical y."""
    lk, device = _lk(), _dev()
    spec = _spec(max_num_loras=4, max_lora_rank=128, rank_choices=(64, 128), kind="fixed",
                 fixed_slots=(3, 0, 2, 1, -1), fixed_lens=(200, 200, 200, 200, 11),
                 hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128)
    raw = sy.emphasize_delta(sy.draw(spec, 54), 40.0)
    outs = []
    for _ in range(3):
        dev = device.prepare(raw, "qkv")
        lk.lora_sgmv_apply(dev["problem"], dev["routing"], dev["workspace"])
        torch.cuda.synchronize()
        assert lk.lora_get_device_status() == 0
        outs.append(device.y_host(dev))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# ------------------------------------------------- seeded random batches --

def _random_case(case):
    """A random small problem for case `case` (seeded): slot count, rank,
    true ranks, widths, request mix (one-token and long requests, base
    requests anywhere before sorting), dtype, layout and options.  Returns
    (raw, kwargs for run_case, projection, run the unsorted form too)."""
    rng = np.random.default_rng(20000 + case)
    R = int(rng.choice([16, 32, 64, 128]))
    S = int(rng.integers(1, 9))
    ranks = sorted({R, max(1, R // 2), int(rng.integers(1, R + 1))})
    hd = int(rng.choice([32, 64]))
    n_heads = int(rng.choice([2, 4, 8]))
    n_kv = int(rng.choice([1, 2])) if n_heads > 2 else 1
    hidden = int(rng.choice([64, 128, 256, 512]))
    n_req = int(rng.integers(1, 11))
    slots = [int(v) for v in rng.integers(-1, S, size=n_req)]
    lens = [int(rng.integers(1, 9)) if rng.random() < 0.5 else
            int(rng.integers(60, 330)) if rng.random() < 0.7 else int(rng.integers(330, 1200)) for _ in range(n_req)]
    dtype = "f32" if rng.random() < 0.15 else "bf16"
    spec = _spec(dtype=dtype, max_num_loras=S, max_lora_rank=R, rank_choices=tuple(ranks), kind="fixed",
                 fixed_slots=tuple(slots), fixed_lens=tuple(lens), hidden=hidden, n_heads=n_heads,
                 n_kv_heads=n_kv, head_dim=hd, rslora_count=int(rng.integers(0, S + 1)))
    raw = sy.draw(spec, 30000 + case)
    if rng.random() < 0.5:
        raw = sy.emphasize_delta(raw, 40.0)
    if rng.random() < 0.3:
        raw = sy.add_bias(raw, case, scale=1.0)
    proj = "qkv" if rng.random() < 0.6 else "o"
    kw = dict(mode="apply" if rng.random() < 0.6 else "split",
              fused=bool(rng.random() < 0.7) or proj == "o")
    if rng.random() < 0.4:
        kw.update(slot_ranks=True, poison=True)
    if rng.random() < 0.3 and kw["mode"] == "apply" and kw["fused"]:
        kw["host_ids"] = True
    unsorted = dtype == "bf16" and rng.random() < 0.3
    return raw, kw, proj, unsorted


@pytest.mark.parametrize("case", range(64))
def test_random_batches(case):
    """Seeded random batches across the kernel families (generic, mma.sync,
    tcgen05, kernels per group), layouts (fused, per projection), options
    (bias, true ranks with NaN in the padding, the routing's host copies,
    rsLoRA slots) and modes (apply, split): every routed row against the
    oracle, rows past `end` bit-identical; some also in arrival order through
    token_rows against the per-token oracle."""
    raw, kw, proj, unsorted = _random_case(case)
    run_case(raw, proj, **kw)
    if unsorted:
        run_unsorted(raw, proj, kw["mode"])
