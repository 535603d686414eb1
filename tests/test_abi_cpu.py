"""The C-ABI library on the host: it loads, exports every entry point the
header declares, and rejects bad arguments before any CUDA call."""
import os
import re

import pytest

import linear_layer_gemms_gb300 as mm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_layer_gemms_gb300 import _build

    _build.build()
    mm.load()


def declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b((?:mmbwd|lnbwd|encbwd)_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported_and_bound():
    names = declared_functions()
    assert "mmbwd_run" in names and "lnbwd_run" in names and "encbwd_run" in names and len(names) >= 14
    lib = mm.load()
    for n in names:
        assert hasattr(lib, n), n
        assert n in mm.SIGNATURES, n
    assert set(mm.SIGNATURES) == set(names)


def test_version_and_strerror():
    assert mm.mmbwd_version() >= 10000
    msgs = {c: mm.strerror(c) for c in range(-11, 1)}
    assert len(set(msgs.values())) == len(msgs)
    assert "unknown" in mm.strerror(-99)


A = 1 << 20  # fake, 16-byte aligned addresses: validation fails before any use


def run(**kw):
    args = dict(dinp=A, dweight=2 * A, dbias=3 * A, dout=4 * A, inp=5 * A, weight=6 * A,
                B=2, T=8, C=64, OC=32, dtype=mm.BF16, stream=0)
    args.update(kw)
    return mm.mmbwd_run(**args)


def test_rejects_bad_dtype_and_shapes():
    assert run(dtype=7) == mm.ERR_DTYPE
    assert run(B=-1) == mm.ERR_SHAPE
    assert run(OC=-8) == mm.ERR_SHAPE
    assert run(B=1 << 40, T=1 << 40) == mm.ERR_SHAPE
    assert run(T=1 << 31) == mm.ERR_SHAPE


def test_rejects_null_misaligned_and_aliased():
    assert run(dout=None) == mm.ERR_NULL
    assert run(dinp=None) == mm.ERR_NULL
    assert run(weight=None) == mm.ERR_NULL
    assert run(inp=A * 5 + 8) == mm.ERR_ALIGN
    assert run(dbias=A * 3 + 2) == mm.ERR_ALIGN
    assert run(C=60) == mm.ERR_ALIGN          # 60 bf16 = 120 bytes, not a multiple of 16
    assert run(OC=36, dtype=mm.BF16) == mm.ERR_ALIGN
    assert run(dinp=4 * A + 64) == mm.ERR_ALIAS    # dinp inside dout
    assert run(dbias=2 * A + 16) == mm.ERR_ALIAS   # dbias inside dweight
    assert run(dweight=A + 32) == mm.ERR_ALIAS     # dweight overlaps dinp


def test_empty_tensors_may_be_null():
    # With B*T == 0 the activations are empty and may be NULL; with no dbias
    # either, the call does no device work at all (safe with fake addresses).
    rc = run(B=0, dinp=None, dout=None, inp=None, dbias=None)
    assert rc in (mm.OK, mm.ERR_CUDA, mm.ERR_ARCH)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU path")
def test_valid_arguments_without_a_gpu_fail_cleanly():
    assert run() in (mm.ERR_CUDA, mm.ERR_ARCH)
    assert mm.mmbwd_device_status()[0] == mm.ERR_CUDA


def test_plan_is_a_pure_function_of_shape():
    for (B, T, C, OC) in [(8, 1024, 768, 3072), (8, 1024, 3072, 768), (8, 1024, 768, 768),
                          (8, 1024, 768, 50304), (4, 1024, 1600, 6400), (1, 5, 8, 16)]:
        a = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        b = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        assert a == b
        BT = B * T
        # CTA pairs: 256-row tiles, 128 or 256 columns per product, an even grid
        assert a["path"] == 1 and 2 <= a["grid"] <= 152 and a["grid"] % 2 == 0
        assert a["tile_n_dinp"] in (128, 256) and a["tile_n_dweight"] in (128, 256)
        assert a["pairs_per_cluster"] in (1, 2) and a["tile_m"] == 256 * a["pairs_per_cluster"]
        assert a["grid"] % (2 * a["pairs_per_cluster"]) == 0
        assert a["dinp_tiles"] == -(-BT // a["tile_m"]) * -(-C // a["tile_n_dinp"])
        assert a["dweight_tiles"] == -(-OC // a["tile_m"]) * -(-C // a["tile_n_dweight"])
        assert a["grid"] // (2 * a["pairs_per_cluster"]) <= a["items"]
        assert a["items"] == a["dinp_tiles"] + a["dweight_tiles"] * a["splits"]
        kb = -(-BT // 64)
        # every split is non-empty and together they cover the reduction
        assert (a["splits"] - 1) * a["kb_per_split"] < kb <= a["splits"] * a["kb_per_split"]
        ws = mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16)
        assert (ws > 0) == (a["splits"] > 1)
    # fp32: three tf32 products on the tensor cores (two products, 256-row
    # tiles, k-blocks of 32) for every shape they take, the tiny check and rows
    # of 4 (mod 8) floats included; the FMA kernel for longer reductions
    f = mm.mmbwd_plan_info(4, 1024, 1600, 6400, mm.F32, 152)
    assert f["path"] == 2 and f["tile_m"] == 256 and f["tile_k"] == 32 and f["grid"] % 2 == 0
    assert f["dinp_tiles"] == -(-4096 // 256) * -(-1600 // f["tile_n_dinp"])
    assert f["dweight_tiles"] == -(-6400 // 256) * -(-1600 // f["tile_n_dweight"])
    assert f["items"] == f["dinp_tiles"] + f["dweight_tiles"]
    assert mm.mmbwd_plan_info(2, 64, 64, 192, mm.F32, 152)["path"] == 2
    assert mm.mmbwd_plan_info(2, 64, 68, 196, mm.F32, 152)["path"] == 2
    assert mm.mmbwd_plan_info(1, 64, 68, 8196, mm.F32, 152)["path"] == 0


def test_split_override_from_environment(monkeypatch):
    monkeypatch.setenv("MMBWD_SPLITK", "3")
    monkeypatch.setenv("MMBWD_GRID", "5")
    a = mm.mmbwd_plan_info(1, 1000, 264, 392, mm.BF16, 152)
    assert a["splits"] == 3 and a["grid"] == 4  # rounded down to whole CTA pairs
    # a forced count that would leave an empty split is lowered, never dropped:
    # 16 k-blocks in 5 splits of 4 would leave the fifth empty, so 4 splits
    monkeypatch.setenv("MMBWD_SPLITK", "5")
    a = mm.mmbwd_plan_info(1, 1024, 264, 392, mm.BF16, 152)
    assert a["splits"] == 4 and a["kb_per_split"] == 4 and a["items"] > 0
    monkeypatch.delenv("MMBWD_SPLITK")
    monkeypatch.delenv("MMBWD_GRID")


def test_one_cta_pair_per_cluster():
    """Every plan runs clusters of one CTA pair (no operand shared across
    pairs), forward and backward, whatever the shape."""
    for shape in ((8, 1024, 768, 3072), (8, 1024, 3072, 768), (8, 1024, 768, 768), (4, 1024, 1600, 6400)):
        a = mm.mmbwd_plan_info(*shape, mm.BF16, 152)
        assert a["pairs_per_cluster"] == 1 and a["tile_m"] == 256 and a["grid"] % 2 == 0


def test_tile_width_override(monkeypatch):
    monkeypatch.setenv("MMBWD_TILE_N", "128,256")
    a = mm.mmbwd_plan_info(8, 1024, 768, 3072, mm.BF16, 152)
    assert (a["tile_n_dinp"], a["tile_n_dweight"]) == (128, 256)
    monkeypatch.setenv("MMBWD_TILE_N", "256,128")
    a = mm.mmbwd_plan_info(8, 1024, 768, 3072, mm.BF16, 152)
    assert (a["tile_n_dinp"], a["tile_n_dweight"]) == (256, 128)


def test_fp32_tensor_core_plans_pair_the_products(monkeypatch):
    """The fp32 tensor-core backward runs both products (and dbias) in one
    launch where their reductions agree on the correction accumulator, else one
    launch each; the operands are split in the kernel, so nothing runs before."""
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    paired = mm.mmbwd_plan_info(4, 1024, 1600, 6400, mm.F32, 152)
    assert paired["path"] == 2 and paired["launches"] == 1 and paired["table"] == 1
    assert paired["items"] == paired["dinp_tiles"] + paired["dweight_tiles"]
    split = mm.mmbwd_plan_info(1, 2560, 264, 512, mm.F32, 152)  # only B*T above the threshold
    assert split["path"] == 2 and split["launches"] == 2
    assert mm.mmbwd_workspace_bytes(4, 1024, 1600, 6400, mm.F32) == 0


def test_workspace_size_formula():
    import os as _os
    _os.environ["MMBWD_SPLITK"] = "2"
    try:
        B, T, C, OC = 1, 1000, 264, 392
        info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        ws = mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16)
        half_tiles = 2 * info["dweight_tiles"]  # per-CTA 128-row parts of the pair tiles
        align = lambda x: (x + 255) // 256 * 256  # noqa: E731
        want = (align(half_tiles * 2 * 128 * info["tile_n_dweight"] * 4) +
                align(2 * -(-OC // info["tile_m"]) * 2 * 128 * 4))
        assert info["launches"] == 2  # the split reduction is a second kernel
        assert ws == want
    finally:
        del _os.environ["MMBWD_SPLITK"]
    assert mm.mmbwd_workspace_bytes(1, 8, 64, 64, mm.F32) == 0
    assert mm.mmbwd_workspace_bytes(-1, 8, 64, 64, mm.BF16) == 0


def test_forward_rejects_bad_arguments():
    f = lambda **kw: mm.mmbwd_forward(**{**dict(out=A, inp=2 * A, weight=3 * A, bias=4 * A, B=2, T=8,  # noqa: E731
                                                 C=64, OC=32, dtype=mm.BF16, stream=0), **kw})
    assert f(dtype=3) == mm.ERR_DTYPE
    assert f(T=-1) == mm.ERR_SHAPE
    assert f(out=None) == mm.ERR_NULL
    assert f(inp=2 * A + 4) == mm.ERR_ALIGN
    assert f(C=12) == mm.ERR_ALIGN
    assert f(out=2 * A + 32) == mm.ERR_ALIAS   # out overlaps inp
    assert f(out=4 * A - 16) == mm.ERR_ALIAS   # out overlaps bias


def test_layernorm_rejects_bad_arguments():
    f = lambda **kw: mm.lnbwd_run(**{**dict(dinp=A, dweight=2 * A, dbias=3 * A, dout=4 * A, inp=5 * A,  # noqa: E731
                                             weight=6 * A, mean=7 * A, rstd=8 * A, B=2, T=8, C=64,
                                             dtype=mm.BF16, stream=0), **kw})
    assert f(dtype=2) == mm.ERR_DTYPE
    assert f(T=-1) == mm.ERR_SHAPE
    assert f(C=(1 << 20) + 8) == mm.ERR_SHAPE            # above LNBWD_MAX_C_BF16
    assert f(C=(1 << 20) + 4, dtype=mm.F32) == mm.ERR_SHAPE  # above LNBWD_MAX_C_F32
    assert f(B=1 << 40, T=1 << 40) == mm.ERR_SHAPE
    assert f(mean=None) == mm.ERR_NULL
    assert f(weight=None) == mm.ERR_NULL
    assert f(dout=None) == mm.ERR_NULL
    assert f(inp=5 * A + 8) == mm.ERR_ALIGN
    assert f(rstd=8 * A + 2) == mm.ERR_ALIGN          # statistics need 4-byte alignment
    assert f(C=60) == mm.ERR_ALIGN                    # 120 bytes per row
    assert f(dinp=4 * A + 64) == mm.ERR_ALIAS         # dinp inside dout
    assert f(dbias=2 * A + 16) == mm.ERR_ALIAS        # dbias overlaps dweight
    assert f(dweight=7 * A) == mm.ERR_ALIAS           # dweight on top of mean
    assert mm.lnbwd_workspace_bytes(-1, 8, 64, mm.BF16) == 0
    assert mm.LNBWD_MAX_C == {mm.F32: 1 << 20, mm.BF16: 1 << 20}


def test_sr_rejects_fp32_and_bad_arguments():
    f = lambda **kw: mm.mmbwd_run_sr(**{**dict(dinp=A, dweight=2 * A, dbias=3 * A, dout=4 * A, inp=5 * A,  # noqa: E731
                                                weight=6 * A, B=2, T=8, C=64, OC=64, dtype=mm.BF16, seed=1,
                                                stream=0), **kw})
    assert f(dtype=mm.F32) == mm.ERR_DTYPE          # stochastic rounding is for bf16 outputs
    assert f(dtype=7) == mm.ERR_DTYPE
    assert f(T=-1) == mm.ERR_SHAPE
    assert f(dout=None) == mm.ERR_NULL
    assert f(dinp=A + 8) == mm.ERR_ALIGN
    assert f(dweight=4 * A) == mm.ERR_ALIAS


def test_encoder_plan_rejects_bad_arguments():
    need = mm.encbwd_plan_bytes(2, 8, 64, 100, mm.BF16)
    assert need > 0 and mm.encbwd_plan_bytes(2, 8, 64, 131072, mm.BF16) == 0
    p = lambda **kw: mm.encbwd_prepare(**{**dict(plan=8 * A, plan_bytes=need, inp=4 * A, B=2, T=8, C=64, V=100,  # noqa: E731
                                                 dtype=mm.BF16, stream=0), **kw})
    assert p(plan=None) == mm.ERR_NULL
    assert p(plan=8 * A + 16) == mm.ERR_ALIGN           # plans are 256-byte aligned
    assert p(plan_bytes=need - 1) == mm.ERR_SHAPE
    assert p(inp=8 * A + 64) == mm.ERR_ALIAS             # ids inside the plan
    assert p(C=12) == mm.ERR_ALIGN
    r = lambda **kw: mm.encbwd_run_planned(**{**dict(dwte=A, dwpe=2 * A, dout=3 * A, plan=8 * A, B=2, T=8,  # noqa: E731
                                                     C=64, V=100, dtype=mm.BF16, seed=None, stream=0), **kw})
    assert r(plan=None) == mm.ERR_NULL
    assert r(plan=8 * A + 32) == mm.ERR_ALIGN
    assert r(dtype=mm.F32, seed=5) == mm.ERR_DTYPE       # stochastic rounding is for bf16 outputs
    assert r(plan=A + 256) == mm.ERR_ALIAS               # plan inside dwte
    assert r(dwpe=3 * A) == mm.ERR_ALIAS


def test_encoder_rejects_bad_arguments():
    f = lambda **kw: mm.encbwd_run(**{**dict(dwte=A, dwpe=2 * A, dout=3 * A, inp=4 * A, B=2, T=8, C=64,  # noqa: E731
                                             V=100, dtype=mm.BF16, stream=0), **kw})
    assert f(dtype=5) == mm.ERR_DTYPE
    assert f(T=-1) == mm.ERR_SHAPE
    assert f(B=2, T=(1 << 23) + 1) == mm.ERR_SHAPE    # above ENCBWD_MAX_POSITIONS
    assert f(V=131072) == mm.ERR_SHAPE                # above ENCBWD_MAX_VOCAB
    assert f(C=65536 + 8) == mm.ERR_SHAPE             # above ENCBWD_MAX_CHANNELS
    assert f(dout=None) == mm.ERR_NULL
    assert f(inp=None) == mm.ERR_NULL
    assert f(dwte=A + 8) == mm.ERR_ALIGN
    assert f(inp=4 * A + 2) == mm.ERR_ALIGN
    assert f(C=12) == mm.ERR_ALIGN                    # 24 bytes per row
    assert f(dwpe=A + 64) == mm.ERR_ALIAS             # dwpe inside dwte
    assert f(dwte=3 * A - 64) == mm.ERR_ALIAS         # dwte runs into dout
    assert mm.encbwd_workspace_bytes(2, 8, 64, 100, mm.BF16) > 0
    assert mm.encbwd_workspace_bytes(-1, 8, 64, 100, mm.BF16) == 0


def test_fp32_tensor_core_path_reduction_limit(monkeypatch):
    """The three-tf32 path's error grows with the reduction length (the tensor
    core rounds each accumulation toward zero), so it is taken only while both
    reduction lengths (OC for dinp, B*T for dweight) are at most 8192, even
    when forced; the forward's is C."""
    monkeypatch.delenv("MMBWD_F32_PATH", raising=False)
    assert mm.mmbwd_plan_info(4, 1024, 1600, 6400, mm.F32, 152)["path"] == 2
    assert mm.mmbwd_plan_info(8, 1024, 768, 8192, mm.F32, 152)["path"] == 2
    assert mm.mmbwd_plan_info(8, 1024, 768, 8200, mm.F32, 152)["path"] == 0
    assert mm.mmbwd_plan_info(16, 1024, 768, 768, mm.F32, 152)["path"] == 0
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    assert mm.mmbwd_plan_info(1, 1024, 512, 16384, mm.F32, 152)["path"] == 0
    assert mm.mmbwd_forward_path(1, 1024, 16384, 512, mm.F32) == 0
    assert mm.mmbwd_forward_path(1, 1024, 8192, 512, mm.F32) == 2
