"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, its host routing builder agrees bit-exactly with the oracle,
and host-side validation rejects bad arguments before touching the GPU."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import adapter_sgmv_lora_gb300 as lk
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_sgmv.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from adapter_sgmv_lora_gb300 import build
    build.build()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert "lora_sgmv_apply" in names and "lora_build_routing" in names
    L = ctypes.CDLL(lk.library_path())
    for n in names:
        assert hasattr(L, n), n


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without liblora_sgmv.so every call raises: there is no CPU fallback."""
    monkeypatch.setattr(lk, "_lib", None)
    monkeypatch.setattr(lk, "LIB_PATH", str(tmp_path / "liblora_sgmv.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        lk.lora_build_routing([0, 1], [1, 1], 2)
    with pytest.raises(RuntimeError, match="no fallback"):
        lk.lora_status_string(0)
    with pytest.raises(RuntimeError, match="no fallback"):
        lk.lib()


def test_status_strings():
    for code, name in lk.STATUS_NAMES.items():
        assert lk.lora_status_string(code).startswith(name)


def _cmp_routing(slots, lens, S):
    a = lk.lora_build_routing(slots, lens, S)
    b = oracle.build_routing(slots, lens, S)
    assert b["status"] == oracle.OK
    for key in ("perm", "lora_ids", "grouped_offsets"):
        assert np.array_equal(a[key], b[key]), key
    for key in ("num_groups", "end", "total_tokens"):
        assert a[key] == b[key], key


@pytest.mark.parametrize("name", ["routing_tiny.json", "routing_unsorted.json"])
def test_routing_golden(name):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", name)))
    r = lk.lora_build_routing(g["req_slot"], g["req_len"], g["max_num_loras"])
    assert r["perm"].tolist() == g["perm"]
    assert r["lora_ids"].tolist() == g["lora_ids"]
    assert r["grouped_offsets"].tolist() == g["grouped_offsets"]
    assert r["end"] == g["end"] and r["total_tokens"] == g["total_tokens"]


def test_routing_matches_oracle_random():
    rng = np.random.default_rng(11)
    for trial in range(400):
        S = int(rng.integers(1, 70))
        n = int(rng.integers(0, 300))
        slots = rng.integers(-1, S, size=n).astype(np.int32)
        lens = rng.integers(0, 40, size=n).astype(np.int32)
        _cmp_routing(slots, lens, S)


def test_routing_matches_oracle_workloads():
    from workloads import synthetic as sy
    for name in sy.SPECS:
        raw = sy.draw(name, 0, with_weights=False) if name != "mixed70b" else None
        if raw is None:
            rng = np.random.default_rng(0)
            slots, lens = sy.draw_requests(rng, sy.SPECS[name])
            _cmp_routing(slots, lens, sy.SPECS[name].max_num_loras)
        else:
            _cmp_routing(raw["req_slot"], raw["req_len"], raw["max_num_loras"])


def test_routing_into_caller_buffers():
    """out_ids / out_offsets receive exactly what the default path returns;
    entries past num_groups are left alone; wrong buffers are refused."""
    rng = np.random.default_rng(12)
    for trial in range(50):
        S = int(rng.integers(1, 40))
        n = int(rng.integers(0, 200))
        slots = rng.integers(-1, S, size=n).astype(np.int32)
        lens = rng.integers(0, 20, size=n).astype(np.int32)
        ref = lk.lora_build_routing(slots, lens, S)
        ids = np.full(S + 3, -7, dtype=np.int32)
        offs = np.full(S + 4, -7, dtype=np.int32)
        got = lk.lora_build_routing(slots, lens, S, out_ids=ids, out_offsets=offs)
        g = ref["num_groups"]
        assert got["num_groups"] == g and got["end"] == ref["end"]
        assert np.array_equal(ids[:g], ref["lora_ids"]) and np.array_equal(offs[:g + 1], ref["grouped_offsets"])
        assert np.array_equal(got["lora_ids"], ref["lora_ids"])
        assert g == 0 or np.shares_memory(got["lora_ids"], ids)
        assert np.all(ids[S:] == -7) and np.all(offs[S + 1:] == -7)
    with pytest.raises(ValueError):
        lk.lora_build_routing([0], [1], 4, out_ids=np.zeros(3, dtype=np.int32))
    with pytest.raises(ValueError):
        lk.lora_build_routing([0], [1], 4, out_offsets=np.zeros(5, dtype=np.int64))


def test_routing_errors():
    with pytest.raises(lk.LoraError) as e:
        lk.lora_build_routing([0, 5], [1, 1], 3)
    assert e.value.status == 4
    with pytest.raises(lk.LoraError) as e:
        lk.lora_build_routing([0], [-3], 3)
    assert e.value.status == 2
    with pytest.raises(lk.LoraError) as e:
        lk.lora_build_routing([0], [1], 0)
    assert e.value.status == 2
    r = lk.lora_build_routing([], [], 5)
    assert r["num_groups"] == 0 and r["end"] == 0


def test_host_validation_without_gpu():
    """Bad problems and routings are rejected on the host with the documented
    codes before any CUDA call (so this runs on a machine with no GPU)."""
    L = lk.lib()
    assert L.lora_shrink(None, None, None, None) == 1
    prob = lk._Problem()
    prob.dtype = 7
    rr = lk._Routing()
    assert L.lora_shrink(ctypes.byref(prob), ctypes.byref(rr), None, None) == 6
    prob.dtype = lk.DTYPE_BF16
    prob.num_tokens, prob.in_dim, prob.max_num_loras, prob.max_lora_rank = 8, 64, 2, 16
    prob.x, prob.x_row_stride, prob.num_slices = 16, 64, 1
    prob.slices[0] = lk._Slice(16, 16 * 64, 16, 16 * 16, 16, 16, 16)
    rr.num_groups, rr.end = 3, 4          # more groups than slots
    assert L.lora_expand(ctypes.byref(prob), ctypes.byref(rr), None, None) == 10
    assert L.lora_last_call_path(None) == 0   # nothing was launched
    rr.num_groups, rr.end = -1, 0         # negative group count
    assert L.lora_expand(ctypes.byref(prob), ctypes.byref(rr), None, None) == 5
    rr.num_groups, rr.end = 1, 9          # end past num_tokens
    assert L.lora_expand(ctypes.byref(prob), ctypes.byref(rr), None, None) == 5
    rr.num_groups, rr.end = 0, 0          # empty routing is a no-op
    assert L.lora_sgmv_apply(ctypes.byref(prob), ctypes.byref(rr), None, 0, None) == 0
    rr.num_groups, rr.end, rr.lora_ids, rr.grouped_offsets = 1, 4, 16, 16
    assert L.lora_sgmv_apply(ctypes.byref(prob), ctypes.byref(rr), None, 0, None) == 8
    # host copies of the triple are checked on the host: offsets must start
    # at 0, not decrease and end at `end`; ids must name slots; the ids need
    # the offsets
    rr.num_groups, rr.end = 2, 4
    ids_ok = np.array([1, 0], dtype=np.int32)
    for offs, ids, code in [([0, 2, 4], None, 8),          # valid: reaches the workspace check
                            ([1, 2, 4], None, 5),          # first offset not 0
                            ([0, 3, 2], None, 5),          # decreasing
                            ([0, 2, 3], None, 5),          # last offset != end
                            ([0, 2, 4], ids_ok, 8),        # valid pair
                            ([0, 2, 4], [0, 2], 4),        # slot 2 of 2
                            ([0, 2, 4], [-1, 0], 4),
                            (None, ids_ok, 1)]:            # ids without offsets
        oh = None if offs is None else np.asarray(offs, dtype=np.int32)
        ih = None if ids is None else np.asarray(ids, dtype=np.int32)
        rr.host_grouped_offsets = None if oh is None else oh.ctypes.data
        rr.host_lora_ids = None if ih is None else ih.ctypes.data
        assert L.lora_sgmv_apply(ctypes.byref(prob), ctypes.byref(rr), None, 0, None) == code, (offs, ids)
    rr.host_grouped_offsets = rr.host_lora_ids = None
    rr.num_groups, rr.end = 1, 4
    prob.slices[0].A_slot_stride = 10     # slot blocks overlap
    assert L.lora_shrink(ctypes.byref(prob), ctypes.byref(rr), 16, None) == 2
    prob.slices[0].A_slot_stride = 16 * 64
    prob.num_slices = 4
    assert L.lora_shrink(ctypes.byref(prob), ctypes.byref(rr), 16, None) == 2
    prob.num_slices = 1
    # set_slot: rank beyond max_lora_rank, slot out of range
    assert L.lora_set_slot(ctypes.byref(prob), 0, 0, 17, 1.0, 0, 16, 16, 0, None) == 3
    assert L.lora_set_slot(ctypes.byref(prob), 0, 2, 4, 1.0, 0, 16, 16, 0, None) == 4
    assert L.lora_set_slot(ctypes.byref(prob), 1, 0, 4, 1.0, 0, 16, 16, 0, None) == 2
    assert L.lora_workspace_bytes(ctypes.byref(prob), 100) == 100 * 16 * 4 + (256 - (6400 % 256)) % 256


def test_token_rows_match_oracle():
    rng = np.random.default_rng(14)
    for _ in range(200):
        S = int(rng.integers(1, 10))
        n = int(rng.integers(0, 40))
        slots = rng.integers(-1, S, size=n).astype(np.int32)
        lens = rng.integers(0, 6, size=n).astype(np.int32)
        r = lk.lora_build_routing(slots, lens, S)
        a = lk.lora_build_token_rows(lens, r["perm"], r["end"])
        b = oracle.token_rows(lens, r["perm"], r["end"])
        assert np.array_equal(a, b)
    with pytest.raises(lk.LoraError):
        lk.lora_build_token_rows([2, 3], [0, 1], 9)   # more rows than the batch has
