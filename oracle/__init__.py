"""ctypes wrapper around the C oracle of matmul_backward (and of the layer's forward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it; the product library never imports it.
``mmbwd_oracle.c`` (the linear layer), ``layernorm_oracle.c`` (the LayerNorm
backward), ``encoder_oracle.c`` (the encoder backward) and ``sr_oracle.c``
(the stochastic-rounding option of the bf16 outputs) state what is computed
and which readings of the pages they take.

Builds (gcc, -O2, -ffp-contract=off, no -ffast-math):
  * ``st``  - single-threaded
  * ``omp`` - the same source with -fopenmp
  * ``mutant<k>`` - the same source with one planted mistake (tests only)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = tuple(os.path.join(_HERE, f)
              for f in ("mmbwd_oracle.c", "layernorm_oracle.c", "encoder_oracle.c", "sr_oracle.c"))
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict = {}

F32, BF16, F64 = 0, 1, 2
DTYPES = {"f32": F32, "bf16": BF16, "f64": F64}
MUTANTS = tuple(range(1, 23))
SR_DINP, SR_DWEIGHT, SR_DBIAS, SR_DWTE, SR_DWPE = 0, 1, 2, 3, 4


def lib_path(variant: str) -> str:
    return os.path.join(_BUILD, f"liboracle_{variant}.so")


def build(variant: str = "st", force: bool = False) -> str:
    """Compile one variant of the oracle and return the path of its .so."""
    out = lib_path(variant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(map(os.path.getmtime, _SRCS)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    flags = ["-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]
    if variant == "omp":
        flags.append("-fopenmp")
    elif variant.startswith("mutant"):
        flags.append(f"-DORACLE_MUTANT={int(variant[6:])}")
    elif variant != "st":
        raise ValueError(variant)
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *flags, *_SRCS, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


class Oracle:
    """One loaded build of the oracle."""

    def __init__(self, variant: str = "st"):
        self.variant = variant
        lib = ctypes.CDLL(build(variant))
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_dinp_rows.argtypes = [vp, vp, i64, vp, vp, vp, i64, i64, i64, ci]
        lib.oracle_dweight_rows.argtypes = [vp, vp, vp, i64, vp, vp, vp, i64, i64, i64, ci]
        lib.oracle_matmul_backward.argtypes = [vp] * 8 + [i64] * 4 + [ci]
        lib.oracle_forward_rows.argtypes = [vp, vp, i64, vp, vp, vp, i64, i64, i64, ci]
        lib.oracle_layernorm_forward.argtypes = [vp] * 6 + [i64, i64, ci]
        lib.oracle_layernorm_dinp_rows.argtypes = [vp, vp, i64] + [vp] * 6 + [ci, i64, i64, ci]
        lib.oracle_layernorm_params.argtypes = [vp] * 8 + [ci, i64, i64, ci]
        lib.oracle_encoder_backward.argtypes = [vp] * 6 + [i64] * 4 + [ci]
        u64 = ctypes.c_uint64
        lib.oracle_splitmix64.argtypes = [u64, u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_sr_draw.argtypes = [u64, ci, i64]
        lib.oracle_sr_draw.restype = ctypes.c_uint32
        lib.oracle_sr_round.argtypes = [vp, vp, i64, u64, ci, i64]
        lib.oracle_sr_round.restype = None
        for f in (lib.oracle_dinp_rows, lib.oracle_dweight_rows, lib.oracle_matmul_backward,
                  lib.oracle_forward_rows, lib.oracle_threads, lib.oracle_mutant,
                  lib.oracle_layernorm_forward, lib.oracle_layernorm_dinp_rows,
                  lib.oracle_layernorm_params, lib.oracle_encoder_backward):
            f.restype = ci
        self._lib = lib

    @property
    def threads(self) -> int:
        return int(self._lib.oracle_threads())

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data

    @staticmethod
    def _check(a, dtype_code):
        if a is None:
            return
        want = {F32: np.float32, BF16: np.uint16, F64: np.float64}[dtype_code]
        assert a.dtype == want and a.flags.c_contiguous, (a.dtype, want)

    def dinp_rows(self, dout, weight, dtype: str, rows=None, dinp_init=None):
        """Rows ``rows`` (all rows if None) of dinp_init + dout @ weight, in float64."""
        dt = DTYPES[dtype]
        BT, OC = dout.shape
        C = weight.shape[1]
        for a in (dout, weight, dinp_init):
            self._check(a, dt)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = BT if r is None else len(r)
        out = np.empty((n, C), dtype=np.float64)
        rc = self._lib.oracle_dinp_rows(out.ctypes.data, self._ptr(r), n, self._ptr(dinp_init),
                                        dout.ctypes.data, weight.ctypes.data, BT, C, OC, dt)
        assert rc == 0
        return out

    def dweight_rows(self, dout, inp, dtype: str, rows=None, dweight_init=None, bias=True):
        """Rows ``rows`` (all if None) of dweight_init + dout^T @ inp and the matching dbias."""
        dt = DTYPES[dtype]
        BT, OC = dout.shape
        C = inp.shape[1]
        for a in (dout, inp, dweight_init):
            self._check(a, dt)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = OC if r is None else len(r)
        out = np.empty((n, C), dtype=np.float64)
        db = np.empty(n, dtype=np.float64) if bias else None
        rc = self._lib.oracle_dweight_rows(out.ctypes.data, self._ptr(db), self._ptr(r), n,
                                           self._ptr(dweight_init), dout.ctypes.data,
                                           inp.ctypes.data, BT, C, OC, dt)
        assert rc == 0
        return out, db

    def forward_rows(self, inp, weight, dtype: str, rows=None, bias=None):
        """Rows ``rows`` (all if None) of inp @ weight^T + bias, in float64."""
        dt = DTYPES[dtype]
        BT, C = inp.shape
        OC = weight.shape[0]
        for a in (inp, weight, bias):
            self._check(a, dt)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = BT if r is None else len(r)
        out = np.empty((n, OC), dtype=np.float64)
        rc = self._lib.oracle_forward_rows(out.ctypes.data, self._ptr(r), n, inp.ctypes.data,
                                           weight.ctypes.data, self._ptr(bias), BT, C, OC, dt)
        assert rc == 0
        return out

    def matmul_backward(self, dout, inp, weight, dtype: str, dinp_init=None, dweight_init=None,
                        bias=True):
        """Full (dinp, dweight, dbias-or-None) in float64; shapes as 2-D (BT, .) arrays."""
        dt = DTYPES[dtype]
        BT, OC = dout.shape
        C = inp.shape[1]
        for a in (dout, inp, weight, dinp_init, dweight_init):
            self._check(a, dt)
        dinp = np.empty((BT, C), dtype=np.float64)
        dweight = np.empty((OC, C), dtype=np.float64)
        dbias = np.empty(OC, dtype=np.float64) if bias else None
        rc = self._lib.oracle_matmul_backward(
            dinp.ctypes.data, dweight.ctypes.data, self._ptr(dbias), dout.ctypes.data,
            inp.ctypes.data, weight.ctypes.data, self._ptr(dinp_init), self._ptr(dweight_init),
            1, BT, C, OC, dt)
        assert rc == 0
        return dinp, dweight, dbias


    # ------------------------------------------------------------------ LayerNorm backward

    def layernorm_forward(self, inp, weight, bias, dtype: str, want_out=True):
        """(out or None, mean, rstd) of the layer norm of each row of ``inp``, in float64."""
        dt = DTYPES[dtype]
        BT, C = inp.shape
        for a in (inp, weight, bias):
            self._check(a, dt)
        out = np.empty((BT, C), dtype=np.float64) if want_out else None
        mean = np.empty(BT, dtype=np.float64)
        rstd = np.empty(BT, dtype=np.float64)
        rc = self._lib.oracle_layernorm_forward(self._ptr(out), mean.ctypes.data, rstd.ctypes.data,
                                                inp.ctypes.data, weight.ctypes.data, self._ptr(bias),
                                                BT, C, dt)
        assert rc == 0
        return out, mean, rstd

    @staticmethod
    def _stat(a):
        code = {np.dtype(np.float32): F32, np.dtype(np.float64): F64}[a.dtype]
        assert a.flags.c_contiguous
        return code

    def layernorm_dinp_rows(self, dout, inp, weight, mean, rstd, dtype: str, rows=None, dinp_init=None):
        """Rows ``rows`` (all if None) of dinp_init + the LayerNorm input gradient, in float64."""
        dt = DTYPES[dtype]
        BT, C = inp.shape
        for a in (dout, inp, weight, dinp_init):
            self._check(a, dt)
        sd = self._stat(mean)
        assert self._stat(rstd) == sd
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = BT if r is None else len(r)
        out = np.empty((n, C), dtype=np.float64)
        rc = self._lib.oracle_layernorm_dinp_rows(out.ctypes.data, self._ptr(r), n, self._ptr(dinp_init),
                                                  dout.ctypes.data, inp.ctypes.data, weight.ctypes.data,
                                                  mean.ctypes.data, rstd.ctypes.data, sd, BT, C, dt)
        assert rc == 0
        return out

    def layernorm_params(self, dout, inp, mean, rstd, dtype: str, dweight_init=None, dbias_init=None):
        """(dweight, dbias) of the LayerNorm backward added to their initial values, in float64."""
        dt = DTYPES[dtype]
        BT, C = inp.shape
        for a in (dout, inp, dweight_init, dbias_init):
            self._check(a, dt)
        sd = self._stat(mean)
        assert self._stat(rstd) == sd
        dw = np.empty(C, dtype=np.float64)
        db = np.empty(C, dtype=np.float64)
        rc = self._lib.oracle_layernorm_params(dw.ctypes.data, db.ctypes.data, self._ptr(dweight_init),
                                               self._ptr(dbias_init), dout.ctypes.data, inp.ctypes.data,
                                               mean.ctypes.data, rstd.ctypes.data, sd, BT, C, dt)
        assert rc == 0
        return dw, db


    # ------------------------------------------------------------------ encoder backward

    def encoder_backward(self, dout, inp, B: int, T: int, V: int, dtype: str, dwte_init=None, dwpe_init=None):
        """(dwte (V, C), dwpe (T, C)) in float64; dout is (B*T, C), inp (B*T,) int32."""
        dt = DTYPES[dtype]
        C = dout.shape[1]
        for a in (dout, dwte_init, dwpe_init):
            self._check(a, dt)
        assert inp.dtype == np.int32 and inp.flags.c_contiguous and inp.size == B * T
        dwte = np.empty((V, C), dtype=np.float64)
        dwpe = np.empty((T, C), dtype=np.float64)
        rc = self._lib.oracle_encoder_backward(dwte.ctypes.data, dwpe.ctypes.data, self._ptr(dwte_init),
                                               self._ptr(dwpe_init), dout.ctypes.data, inp.ctypes.data,
                                               B, T, C, V, dt)
        if rc == -2:
            raise ValueError("token id outside [0, V)")
        assert rc == 0
        return dwte, dwpe


    # ------------------------------------------------------------------ stochastic rounding
    def splitmix64(self, seed: int, n: int) -> int:
        """The n-th output (from 0) of splitmix64 seeded with ``seed``."""
        return int(self._lib.oracle_splitmix64(seed, n))

    def sr_draw(self, seed: int, tensor: int, e: int) -> int:
        return int(self._lib.oracle_sr_draw(seed, tensor, e))

    def sr_round(self, values, seed: int, tensor: int, e0: int = 0):
        """bf16 bit patterns (uint16, same shape) of float64 ``values`` rounded
        stochastically; element i of the flattened array has index e0 + i."""
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        self._lib.oracle_sr_round(v.ctypes.data, out.ctypes.data, v.size, seed, tensor, e0)
        return out

    def matmul_backward_sr(self, dout, inp, weight, seed: int, dinp_init=None, dweight_init=None, bias=True):
        """mmbwd_run_sr's outputs (bf16 bit patterns): the exact results of
        matmul_backward, each rounded stochastically as a float."""
        dinp, dweight, dbias = self.matmul_backward(dout, inp, weight, "bf16", dinp_init, dweight_init, bias)
        return (self.sr_round(dinp, seed, SR_DINP), self.sr_round(dweight, seed, SR_DWEIGHT),
                None if dbias is None else self.sr_round(dbias, seed, SR_DBIAS))

    def encoder_backward_sr(self, dout, inp, B: int, T: int, V: int, seed: int, dwte_init=None, dwpe_init=None):
        """encbwd_run_sr's outputs (bf16 bit patterns): the exact results of
        encoder_backward, each rounded stochastically as a float."""
        dwte, dwpe = self.encoder_backward(dout, inp, B, T, V, "bf16", dwte_init, dwpe_init)
        return self.sr_round(dwte, seed, SR_DWTE), self.sr_round(dwpe, seed, SR_DWPE)


def get(variant: str = "st") -> Oracle:
    with _lock:
        if variant not in _libs:
            _libs[variant] = Oracle(variant)
        return _libs[variant]
