"""lora_sgmv_apply_noalloc: the entry point for callers that cannot allocate
device memory (a plug-in inside a host framework that owns every device
allocation, or a latency-critical loop where an allocation could stall).

It must give the same y as lora_sgmv_apply with a caller-provided workspace,
within the bf16 tolerance of the parity tests, on two calls in a row (the
second call reuses the fixed in-library array that the first call left
filled), and the same y as the CPU oracle on every shape family it takes:
decode-sized batches, long rank-64 groups, the general kernels (true ranks,
a bias) called right after a larger call that left its intermediate in the
array, and fp32.  This file is collected last so that a run stopping at the
first failure has already run every other test; it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import synthetic as sy

pytestmark = pytest.mark.gpu

TOL_Y = {"bf16": 2e-2, "f32": 1e-3}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()


def _to_f64(y):
    return y.detach().float().double().cpu().numpy()


def _check_against_oracle(raw, proj, dev, slot_ranks=False):
    """Every routed row of dev's y against the oracle; rows >= end unchanged."""
    from workloads import device
    ref = oracle.prepare_problem(raw, proj)
    end = ref["end"]
    assert dev["route_host"]["end"] == end
    got = oracle.to_f64(device.y_host(dev), raw["dtype"])
    y_in = oracle.to_f64(raw["y_" + proj], raw["dtype"])
    assert np.array_equal(got[end:], y_in[end:])
    if end == 0:
        return
    _, ys = oracle.problem_rows(ref, np.arange(end, dtype=np.int32))
    col = 0
    for yj in ys:
        g = got[:end, col:col + yj.shape[1]]
        err = np.abs(g - yj) / (1.0 + np.abs(yj))
        assert err.max() <= TOL_Y[raw["dtype"]], (proj, float(err.max()))
        col += yj.shape[1]


def test_noalloc_matches_apply_two_calls_in_a_row():
    import adapter_sgmv_lora_gb300 as lk
    from workloads import device

    for seed, proj in ((0, "qkv"), (1, "o")):
        raw = sy.draw("decode8b", seed)
        ref = device.prepare(raw, proj)   # existing entry point, own workspace
        got = device.prepare(raw, proj)   # new entry point, no workspace
        assert torch.equal(ref["y_all"], got["y_all"])
        lk.lora_sgmv_apply(ref["problem"], ref["routing"], ref["workspace"])
        lk.lora_sgmv_apply_noalloc(got["problem"], got["routing"])
        torch.cuda.synchronize()
        assert lk.lora_get_device_status() == 0
        a, b = _to_f64(ref["y_all"]), _to_f64(got["y_all"])
        err = np.abs(b - a) / (1.0 + np.abs(a))
        assert err.max() <= TOL_Y["bf16"], (proj, float(err.max()))
        end = ref["route_host"]["end"]
        assert end > 0
        # rows at or past end untouched by either call
        y0 = device.storage_to_torch(raw["y_" + proj], "bf16")
        assert torch.equal(got["y_all"][end:], y0[end:])
        _check_against_oracle(raw, proj, got)


def test_noalloc_long_rank64_groups_against_oracle():
    """Long groups at rank 64 (which lora_sgmv_apply sends to the tensor-core
    kernels) go through the static array on the cluster mma.sync shrink and
    the mma.sync expand: every routed row against the oracle."""
    import adapter_sgmv_lora_gb300 as lk
    from workloads import device

    spec = sy.custom_spec(max_num_loras=4, max_lora_rank=64, rank_choices=(32, 64), kind="fixed",
                          fixed_slots=(2, 0, 3, 1, -1), fixed_lens=(300, 129, 513, 200, 9), hidden=1024,
                          n_heads=16, n_kv_heads=4, head_dim=64)
    raw = sy.draw(spec, 5)
    for proj in ("qkv", "o"):
        dev = device.prepare(raw, proj)
        lk.lora_sgmv_apply_noalloc(dev["problem"], dev["routing"])
        bits, _ = lk.lora_last_call_path()
        assert bits == lk.PATH_MMA_SHRINK | lk.PATH_MMA_EXPAND, hex(bits)
        torch.cuda.synchronize()
        assert lk.lora_get_device_status() == 0
        _check_against_oracle(raw, proj, dev)


def test_noalloc_general_kernels_after_a_larger_call():
    """A large call leaves its intermediate in the shared array; a smaller
    call on the general kernels (true ranks with NaN past them, a bias) must
    still read only what it wrote itself."""
    import adapter_sgmv_lora_gb300 as lk
    from workloads import device

    big = sy.draw("prefill8b", 3)
    dev_big = device.prepare(big, "qkv")
    end_big = dev_big["route_host"]["end"]
    assert end_big * 3 * 64 * 4 > 8 * 2 ** 20  # fills more than half the array
    lk.lora_sgmv_apply_noalloc(dev_big["problem"], dev_big["routing"])
    raw = sy.add_bias(sy.draw("decode8b", 6), 6)
    dev = device.prepare(raw, "qkv", slot_ranks=True)
    R = raw["max_lora_rank"]
    for s, r in enumerate(raw["rank"]):  # NaN in the padding past ceil16(rank): never read
        k16 = min(R, (int(r) + 15) // 16 * 16)
        if k16 < R:
            for j in range(3):
                dev["stacks"]["A"][s, j * R + k16:(j + 1) * R].fill_(float("nan"))
            dev["stacks"]["B"][s, :, k16:].fill_(float("nan"))
    lk.lora_sgmv_apply_noalloc(dev["problem"], dev["routing"])
    torch.cuda.synchronize()
    assert lk.lora_get_device_status() == 0
    _check_against_oracle(raw, "qkv", dev)


def test_noalloc_fp32_against_oracle():
    import adapter_sgmv_lora_gb300 as lk
    from workloads import device

    for proj in ("qkv", "o"):
        raw = sy.draw("tiny", 0)
        dev = device.prepare(raw, proj)
        lk.lora_sgmv_apply_noalloc(dev["problem"], dev["routing"])
        bits, _ = lk.lora_last_call_path()
        assert bits == lk.PATH_GENERIC_SHRINK | lk.PATH_GENERIC_EXPAND, hex(bits)
        torch.cuda.synchronize()
        assert lk.lora_get_device_status() == 0
        _check_against_oracle(raw, proj, dev)


def test_noalloc_rejects_batches_beyond_its_array():
    import adapter_sgmv_lora_gb300 as lk
    from workloads import device

    # 12 000 routed rows x 3 slices x rank 128 x 4 bytes = 18.4 MB > 16 MiB
    spec = sy.custom_spec(hidden=128, n_heads=4, n_kv_heads=4, head_dim=32, max_num_loras=1,
                          max_lora_rank=128, rank_choices=(128,), kind="fixed",
                          fixed_slots=(0,) * 12, fixed_lens=(1000,) * 12)
    dev = device.prepare(sy.draw(spec, 0), "qkv")
    need = lk.lora_workspace_bytes(dev["problem"], dev["route_host"]["end"])
    assert need > lk.NOALLOC_MAX_WORKSPACE_BYTES
    before = dev["y_all"].clone()
    with pytest.raises(lk.LoraError) as e:
        lk.lora_sgmv_apply_noalloc(dev["problem"], dev["routing"])
    assert e.value.status == 8  # LORA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(dev["y_all"], before)
