"""lora_sgmv_apply_noalloc: the entry point for callers that cannot allocate
device memory (a plug-in inside a host framework that owns every device
allocation, or a latency-critical loop where an allocation could stall).

It must give the same y as lora_sgmv_apply with a caller-provided workspace,
within the bf16 tolerance of the parity tests, on two calls in a row (the
second call reuses the fixed in-library array that the first call left
filled).  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest
import torch

from workloads import synthetic as sy

pytestmark = pytest.mark.gpu

TOL_Y = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()


def _to_f64(y):
    return y.detach().float().double().cpu().numpy()


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
        assert err.max() <= TOL_Y, (proj, float(err.max()))
        end = ref["route_host"]["end"]
        assert end > 0
        # rows at or past end untouched by either call
        y0 = device.storage_to_torch(raw["y_" + proj], "bf16")
        assert torch.equal(got["y_all"][end:], y0[end:])


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
