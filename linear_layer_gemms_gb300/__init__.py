"""GB300 (sm_103a) backward pass of a GPT-2 linear layer.

Thin Python binding of the C-ABI library ``libmmbwd.so`` (declared in
``include/mmbwd.h``): the same entry points, arguments marshalled through
ctypes, nothing computed here. Every step of the backward pass runs in the
library's CUDA kernels; if the library is not built this module raises on
first use instead of falling back to anything else.

    dinp    (B,T,C)  += dout . weight
    dweight (OC,C)   += dout^T . inp
    dbias   (OC)      = sum over (b,t) of dout        (NULL / None skips it)

and the layer's forward, out = inp . weight^T + bias (mmbwd_forward); plus the
LayerNorm backward of a GPT-2 block (lnbwd_run, include/layernorm_backward.h)
and the encoder backward (encbwd_run, include/encoder_backward.h).

Pointers may be given as integers or as objects with ``data_ptr()`` (for
example torch tensors on the current CUDA device); ``stream`` is a raw
``cudaStream_t`` integer, or None for the current torch stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

F32 = 0
BF16 = 1

OK = 0
ERR_NULL, ERR_DTYPE, ERR_SHAPE, ERR_ALIGN, ERR_ALIAS = -1, -2, -3, -4, -5
ERR_ALLOC, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_ARCH, ERR_CAPTURE = -6, -7, -8, -9, -10
ERR_SCRATCH, ERR_MEMORY = -11, -12
STATIC_SCRATCH_BYTES = 32 << 20  # MMBWD_STATIC_SCRATCH_BYTES

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmmbwd.so")

# Names and C signatures of every entry point declared in include/mmbwd.h,
# include/layernorm_backward.h and include/encoder_backward.h.
_vp, _i64, _ci, _u64, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                             ctypes.c_size_t)
SIGNATURES = {
    "mmbwd_run": ([_vp] * 6 + [_i64] * 4 + [_ci, _vp], _ci),
    "mmbwd_run_sr": ([_vp] * 6 + [_i64] * 4 + [_ci, _u64, _vp], _ci),
    "mmbwd_workspace_bytes": ([_i64] * 4 + [_ci], _sz),
    "mmbwd_release": ([], _ci),
    "mmbwd_strerror": ([_ci], ctypes.c_char_p),
    "mmbwd_device_status": ([_ci, ctypes.POINTER(_ci)], _ci),
    "mmbwd_version": ([], _ci),
    "mmbwd_plan_info": ([_i64] * 4 + [_ci, _ci, ctypes.POINTER(_ci), _ci], _ci),
    "mmbwd_selftest_wait_timeout": ([_u64], _ci),
    "mmbwd_debug_fail_next_alloc": ([_ci], None),
    "mmbwd_debug_fail_next_launch": ([_ci], None),
    "mmbwd_run_static_scratch": ([_vp] * 6 + [_i64] * 4 + [_ci, _vp], _ci),
    "mmbwd_forward": ([_vp] * 4 + [_i64] * 4 + [_ci, _vp], _ci),
    "mmbwd_forward_path": ([_i64] * 4 + [_ci], _ci),
    "lnbwd_run": ([_vp] * 8 + [_i64] * 3 + [_ci, _vp], _ci),
    "encbwd_run": ([_vp] * 4 + [_i64] * 4 + [_ci, _vp], _ci),
    "encbwd_run_sr": ([_vp] * 4 + [_i64] * 4 + [_ci, _u64, _vp], _ci),
    "encbwd_plan_bytes": ([_i64] * 4 + [_ci], _sz),
    "encbwd_prepare": ([_vp, _sz, _vp] + [_i64] * 4 + [_ci, _vp], _ci),
    "encbwd_run_planned": ([_vp] * 4 + [_i64] * 4 + [_ci, ctypes.POINTER(_u64), _vp], _ci),
    "encbwd_workspace_bytes": ([_i64] * 4 + [_ci], _sz),
    "lnbwd_workspace_bytes": ([_i64] * 3 + [_ci], _sz),
}
LNBWD_MAX_C = {F32: 1 << 20, BF16: 1 << 20}  # LNBWD_MAX_C_F32, LNBWD_MAX_C_BF16
ENCBWD_MAX_POSITIONS, ENCBWD_MAX_VOCAB, ENCBWD_MAX_CHANNELS = 1 << 24, 131071, 65536

_lock = threading.Lock()
_lib = None


class MmbwdError(RuntimeError):
    def __init__(self, code: int, what: str = "mmbwd"):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


def load(path: str | None = None):
    """Load libmmbwd.so (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libmmbwd.so is not built ({p}); run __graft_entry__.build()")
            lib = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is not None:
        return int(stream)
    import torch  # only for the current stream handle

    return torch.cuda.current_stream().cuda_stream


def mmbwd_run(dinp, dweight, dbias, dout, inp, weight, B: int, T: int, C: int, OC: int, dtype: int,
              stream=None) -> int:
    """Enqueue one backward pass; returns the C status code (0 = OK)."""
    return load().mmbwd_run(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout), _ptr(inp),
                            _ptr(weight), B, T, C, OC, dtype, _stream(stream))


def mmbwd_run_sr(dinp, dweight, dbias, dout, inp, weight, B: int, T: int, C: int, OC: int, dtype: int,
                 seed: int, stream=None) -> int:
    """mmbwd_run with the bf16 outputs rounded stochastically (unbiased; the
    threshold of each element comes from the splitmix64 generator seeded with
    ``seed``, so the same seed repeats the same bits). bf16 only."""
    return load().mmbwd_run_sr(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout), _ptr(inp),
                               _ptr(weight), B, T, C, OC, dtype, seed, _stream(stream))


def mmbwd_run_static_scratch(dinp, dweight, dbias, dout, inp, weight, B: int, T: int, C: int, OC: int,
                             dtype: int, stream=None) -> int:
    """Like mmbwd_run, but never allocates device memory: for callers that
    cannot (inside an allocator callback, under a fixed memory budget, or in a
    runtime that forbids cudaMalloc once running). Its split reduction uses the
    library's fixed STATIC_SCRATCH_BYTES buffer, shared by every call on the
    device, so overlapping calls race; larger needs return ERR_SCRATCH."""
    return load().mmbwd_run_static_scratch(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout),
                                           _ptr(inp), _ptr(weight), B, T, C, OC, dtype,
                                           _stream(stream))


def mmbwd_forward(out, inp, weight, bias, B: int, T: int, C: int, OC: int, dtype: int,
                  stream=None) -> int:
    """Enqueue out = inp . weight^T + bias (bias may be None); returns the status."""
    return load().mmbwd_forward(_ptr(out), _ptr(inp), _ptr(weight), _ptr(bias), B, T, C, OC, dtype,
                                _stream(stream))


def lnbwd_run(dinp, dweight, dbias, dout, inp, weight, mean, rstd, B: int, T: int, C: int, dtype: int,
              stream=None) -> int:
    """Enqueue the LayerNorm backward (dinp, dweight and dbias all +=); mean
    and rstd are fp32 row statistics; returns the C status code."""
    return load().lnbwd_run(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout), _ptr(inp), _ptr(weight),
                            _ptr(mean), _ptr(rstd), B, T, C, dtype, _stream(stream))


def encbwd_run(dwte, dwpe, dout, inp, B: int, T: int, C: int, V: int, dtype: int, stream=None) -> int:
    """Enqueue the encoder backward (dwte and dwpe +=); inp holds int32 token
    ids; returns the C status code."""
    return load().encbwd_run(_ptr(dwte), _ptr(dwpe), _ptr(dout), _ptr(inp), B, T, C, V, dtype, _stream(stream))


def encbwd_run_sr(dwte, dwpe, dout, inp, B: int, T: int, C: int, V: int, dtype: int, seed: int,
                  stream=None) -> int:
    """encbwd_run with the bf16 outputs rounded stochastically (seeded, as
    mmbwd_run_sr); bf16 only."""
    return load().encbwd_run_sr(_ptr(dwte), _ptr(dwpe), _ptr(dout), _ptr(inp), B, T, C, V, dtype, seed,
                                _stream(stream))


def encbwd_plan_bytes(B: int, T: int, C: int, V: int, dtype: int) -> int:
    """Bytes of the device buffer encbwd_prepare fills (0 for invalid arguments)."""
    return int(load().encbwd_plan_bytes(B, T, C, V, dtype))


def encbwd_prepare(plan, plan_bytes: int, inp, B: int, T: int, C: int, V: int, dtype: int, stream=None) -> int:
    """Sort the token ids into ``plan`` (device, 256-byte aligned): the part of
    the encoder backward that depends only on inp, to run ahead of time."""
    return load().encbwd_prepare(_ptr(plan), plan_bytes, _ptr(inp), B, T, C, V, dtype, _stream(stream))


def encbwd_run_planned(dwte, dwpe, dout, plan, B: int, T: int, C: int, V: int, dtype: int, seed=None,
                       stream=None) -> int:
    """dwte and dwpe += from a prepared plan (one launch); ``seed`` (an int)
    selects stochastic rounding of bf16 outputs, None rounds to nearest."""
    s = None if seed is None else ctypes.byref(_u64(seed))
    return load().encbwd_run_planned(_ptr(dwte), _ptr(dwpe), _ptr(dout), _ptr(plan), B, T, C, V, dtype, s,
                                     _stream(stream))


def encbwd_workspace_bytes(B: int, T: int, C: int, V: int, dtype: int) -> int:
    return int(load().encbwd_workspace_bytes(B, T, C, V, dtype))


def lnbwd_workspace_bytes(B: int, T: int, C: int, dtype: int) -> int:
    return int(load().lnbwd_workspace_bytes(B, T, C, dtype))


def mmbwd_forward_path(B: int, T: int, C: int, OC: int, dtype: int) -> int:
    """0 = fp32 FMA kernel, 1 = bf16 tensor cores, 2 = fp32 from three tf32 products."""
    return int(load().mmbwd_forward_path(B, T, C, OC, dtype))


def mmbwd_workspace_bytes(B: int, T: int, C: int, OC: int, dtype: int) -> int:
    return int(load().mmbwd_workspace_bytes(B, T, C, OC, dtype))


def mmbwd_release() -> int:
    return load().mmbwd_release()


def strerror(code: int) -> str:
    return load().mmbwd_strerror(code).decode()


def mmbwd_strerror(code: int) -> str:
    return strerror(code)


def mmbwd_device_status(reset: bool = True):
    """(status, [block, wait site, item]) of the device status word."""
    info = (ctypes.c_int * 3)()
    code = load().mmbwd_device_status(1 if reset else 0, info)
    return code, list(info)


def mmbwd_version() -> int:
    return load().mmbwd_version()


PLAN_FIELDS = ("path", "grid", "items", "splits", "kb_per_split", "dinp_tiles", "dweight_tiles",
               "table", "tile_m", "tile_n_dinp", "tile_n_dweight", "tile_k", "stages", "launches",
               "pairs_per_cluster")


def mmbwd_plan_info(B: int, T: int, C: int, OC: int, dtype: int, num_sms: int = 0) -> dict:
    out = (ctypes.c_int * len(PLAN_FIELDS))()
    n = load().mmbwd_plan_info(B, T, C, OC, dtype, num_sms, out, len(PLAN_FIELDS))
    if n < 0:
        raise MmbwdError(n, "mmbwd_plan_info")
    return dict(zip(PLAN_FIELDS, list(out)[:n]))


def mmbwd_selftest_wait_timeout(timeout_ns: int) -> int:
    return load().mmbwd_selftest_wait_timeout(timeout_ns)


def mmbwd_debug_fail_next_alloc(n: int) -> None:
    load().mmbwd_debug_fail_next_alloc(n)


def mmbwd_debug_fail_next_launch(n: int) -> None:
    load().mmbwd_debug_fail_next_launch(n)


def matmul_backward(dinp, dweight, dbias, dout, inp, weight, stream=None) -> None:
    """Convenience wrapper for torch tensors: shapes from the tensors, dtype
    from their element type (float32 or bfloat16); raises MmbwdError on a
    non-zero status."""
    import torch

    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(dout.dtype)
    if dt is None:
        raise MmbwdError(ERR_DTYPE, "matmul_backward")
    if dout.dim() == 3:
        B, T, OC = dout.shape
    else:
        (BT, OC), B = dout.shape, 1
        T = BT
    C = inp.shape[-1]
    rc = mmbwd_run(dinp, dweight, dbias, dout, inp, weight, B, T, C, OC, dt, stream)
    if rc != OK:
        raise MmbwdError(rc, "mmbwd_run")
