"""Planner invariants over many shapes (host only, no GPU): every plan the
C ABI reports for seeded random GPT-style shapes is internally consistent --
tile counts, items and splits add up, the grid is an even number of CTAs no
larger than the work, every split is non-empty -- and the fp32 tensor-core
backward runs its two products in one launch exactly when their reduction
lengths agree on the correction accumulator."""
import numpy as np

import linear_layer_gemms_gb300 as mm

CORR_K = 2048  # reductions longer than this keep the fp32 correction products apart


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        B = int(rng.integers(1, 9))
        T = int(rng.integers(1, 2049))
        C = 8 * int(rng.integers(1, 1025))
        OC = 8 * int(rng.integers(1, 4097))
        yield B, T, C, OC


def test_bf16_plans_are_consistent():
    for B, T, C, OC in _shapes(300, 11):
        a = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        BT = B * T
        assert a["path"] == 1 and a["launches"] in (1, 2)
        assert 2 <= a["grid"] <= 152 and a["grid"] % 2 == 0
        assert a["tile_n_dinp"] in (128, 256) and a["tile_n_dweight"] in (128, 256)
        assert a["dinp_tiles"] == -(-BT // 256) * -(-C // a["tile_n_dinp"])
        assert a["dweight_tiles"] == -(-OC // 256) * -(-C // a["tile_n_dweight"])
        assert a["items"] == a["dinp_tiles"] + a["dweight_tiles"] * a["splits"]
        assert a["grid"] // 2 <= a["items"]
        kb = -(-BT // 64)
        assert 1 <= a["splits"] <= 16
        assert (a["splits"] - 1) * a["kb_per_split"] < kb <= a["splits"] * a["kb_per_split"]
        assert (a["launches"] == 2) == (a["splits"] > 1)
        ws = mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16)
        assert (ws > 0) == (a["splits"] > 1)


def test_fp32_tensor_core_plans_are_consistent(monkeypatch):
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    seen = set()
    for B, T, C, OC in _shapes(300, 12):
        a = mm.mmbwd_plan_info(B, T, C, OC, mm.F32, 152)
        BT = B * T
        if a["path"] != 2:  # shapes the split layout cannot take run on the FMA kernel
            assert a["path"] == 0
            continue
        assert a["tile_m"] == 256 and a["tile_k"] == 32 and a["grid"] % 2 == 0 and a["grid"] <= 152
        assert a["dinp_tiles"] == -(-BT // 256) * -(-C // a["tile_n_dinp"])
        assert a["dweight_tiles"] == -(-OC // 256) * -(-C // a["tile_n_dweight"])
        assert a["items"] == a["dinp_tiles"] + a["dweight_tiles"]
        paired = (OC > CORR_K) == (BT > CORR_K) and a["items"] <= 3072
        assert a["launches"] == (1 if paired else 2)
        if paired:
            assert a["tile_n_dinp"] == a["tile_n_dweight"] and a["table"] == 1
        seen.add(a["launches"])
    assert seen == {1, 2}  # both kinds of plan occur among the shapes


def test_fp32_needs_no_workspace(monkeypatch):
    # the tensor-core path splits the raw operands in shared memory and forms
    # dbias in the same launch; the FMA kernel works in place
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    for B, T, C, OC in [(4, 1024, 1600, 6400), (1, 301, 264, 136), (2, 777, 392, 520), (8, 1024, 768, 3072)]:
        assert mm.mmbwd_plan_info(B, T, C, OC, mm.F32, 152)["path"] == 2
        assert mm.mmbwd_workspace_bytes(B, T, C, OC, mm.F32) == 0


def test_forced_split_length(monkeypatch):
    # MMBWD_SPLIT_KB fixes the k-blocks per split; the last split takes the rest
    B, T, C, OC = 8, 1024, 768, 768  # 128 k-blocks of B*T
    for kps in (20, 43, 64, 100, 128):
        monkeypatch.setenv("MMBWD_SPLIT_KB", str(kps))
        a = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        assert a["kb_per_split"] == kps and a["splits"] == -(-128 // kps)
        assert (a["launches"] == 2) == (a["splits"] > 1)
    monkeypatch.delenv("MMBWD_SPLIT_KB")
    # the planner's own choice for GPT-2 small qkv: a long split and a short one
    a = mm.mmbwd_plan_info(8, 1024, 768, 2304, mm.BF16, 152)
    assert a["splits"] == 2 and a["kb_per_split"] > 64
