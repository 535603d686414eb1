"""Seeded synthetic inputs for the matmul_backward workloads.

This package draws the random inputs that both the CPU oracle and the CUDA
path consume. It contains no arithmetic of the backward pass itself: only the
counter-based generator in ``gen.c`` (splitmix64 words, Box-Muller normals,
round-to-nearest-even to f32/bf16) and the workload recipes below.

bf16 tensors are returned as ``numpy.uint16`` arrays holding the raw bit
patterns; ``bf16_bits_to_f64`` converts them exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
_DT = {"f32": F32, "bf16": BF16, "f64": F64}
_NP = {F32: np.float32, BF16: np.uint16, F64: np.float64}

# Per-tensor stream ids; a layer index adds 16 * layer so that two layers of
# one workload draw independent values.
STREAM = {"inp": 1, "weight": 2, "dout": 3, "dinp_init": 4, "dweight_init": 5, "dbias_init": 6,
          "lm_index": 7}


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libsynth.so with gcc (OpenMP on)."""
    src = os.path.join(_HERE, "gen.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", src, "-o", tmp,
                           "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, dbl, vp, ci = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_double,
                                     ctypes.c_void_p, ctypes.c_int)
            lib.synth_normal.argtypes = [vp, i64, ci, u64, u64, dbl, dbl]
            lib.synth_normal.restype = ci
            lib.synth_lmhead_dout.argtypes = [vp, i64, i64, ci, u64, u64, u64, dbl, dbl]
            lib.synth_lmhead_dout.restype = ci
            lib.synth_lmhead_hot_index.argtypes = [i64, i64, u64, u64]
            lib.synth_lmhead_hot_index.restype = i64
            lib.synth_uniform.argtypes = [vp, i64, u64, u64]
            lib.synth_uniform.restype = ci
            _lib = lib
    return _lib


def normal(shape, dtype: str, seed: int, stream: int, mean: float = 0.0, std: float = 1.0,
           out: np.ndarray | None = None) -> np.ndarray:
    """mean + std * N(0,1), drawn from (seed, stream), rounded to ``dtype``."""
    dt = _DT[dtype]
    n = int(np.prod(shape)) if len(shape) else 1
    if out is None:
        out = np.empty(shape, dtype=_NP[dt])
    assert out.dtype == _NP[dt] and out.flags.c_contiguous and out.size == n
    rc = _load().synth_normal(out.ctypes.data, n, dt, seed, stream, mean, std)
    assert rc == 0
    return out


def lmhead_dout(rows: int, cols: int, dtype: str, seed: int, stream_noise: int, stream_index: int,
                std: float, spike: float, out: np.ndarray | None = None) -> np.ndarray:
    """Dense std*N(0,1) plus one ``spike`` per row at a uniform random column."""
    dt = _DT[dtype]
    if out is None:
        out = np.empty((rows, cols), dtype=_NP[dt])
    rc = _load().synth_lmhead_dout(out.ctypes.data, rows, cols, dt, seed, stream_noise, stream_index,
                                   std, spike)
    assert rc == 0
    return out


def lmhead_hot_index(row: int, cols: int, seed: int, stream_index: int) -> int:
    return int(_load().synth_lmhead_hot_index(row, cols, seed, stream_index))


def uniform(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    assert _load().synth_uniform(out.ctypes.data, n, seed, stream) == 0
    return out


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f64(a) if dtype == "bf16" else a.astype(np.float64)


# ---------------------------------------------------------------------------
# Workload recipes (shapes and value distributions of the GPT-2 linear layers)
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Layer:
    """One linear layer's backward problem: inp (B,T,C), weight (OC,C), dout (B,T,OC)."""
    name: str
    B: int
    T: int
    C: int
    OC: int
    dtype: str            # storage type of all six tensors: "f32" or "bf16"
    bias: bool            # whether dbias is requested
    inp_std: float = 1.0
    w_std: float = 0.02
    dout_std: float = 1e-2
    init_std: float = 0.0  # std of the dinp/dweight pre-fill (0: start at zero)
    dout_kind: str = "normal"  # or "lmhead"
    layer: int = 0         # stream offset index

    @property
    def BT(self) -> int:
        return self.B * self.T

    def flops(self) -> int:
        """4*B*T*C*OC for the two products, plus B*T*OC adds for the bias sum."""
        f = 4 * self.BT * self.C * self.OC
        return f + (self.BT * self.OC if self.bias else 0)

    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


@dataclass
class Workload:
    name: str
    layers: list = field(default_factory=list)

    def flops(self) -> int:
        return sum(l.flops() for l in self.layers)


def _gpt2(name, B, T, C, OC, dtype, bias=True, layer=0, **kw):
    return Layer(name, B, T, C, OC, dtype, bias, layer=layer, **kw)


WORKLOADS = {
    # fp32 check with += pre-fill
    "tiny": Workload("tiny", [_gpt2("tiny", 2, 64, 64, 192, "f32", dout_std=1.0, init_std=0.01)]),
    "attn_proj": Workload("attn_proj", [_gpt2("attn_proj", 8, 1024, 768, 768, "bf16")]),
    "qkv": Workload("qkv", [_gpt2("qkv", 8, 1024, 768, 2304, "bf16")]),
    # the headline: the two MLP linears of one GPT-2 small block
    "mlp": Workload("mlp", [_gpt2("mlp_fc", 8, 1024, 768, 3072, "bf16", layer=0),
                            _gpt2("mlp_fc_proj", 8, 1024, 3072, 768, "bf16", layer=1)]),
    "lm_head": Workload("lm_head", [_gpt2("lm_head", 8, 1024, 768, 50304, "bf16", bias=False,
                                          dout_kind="lmhead", dout_std=1e-4)]),
    "xl_fc_bf16": Workload("xl_fc_bf16", [_gpt2("xl_fc", 4, 1024, 1600, 6400, "bf16")]),
    "xl_qkv_bf16": Workload("xl_qkv_bf16", [_gpt2("xl_qkv", 4, 1024, 1600, 4800, "bf16")]),
    "xl_fc_f32": Workload("xl_fc_f32", [_gpt2("xl_fc", 4, 1024, 1600, 6400, "f32")]),
    "xl_qkv_f32": Workload("xl_qkv_f32", [_gpt2("xl_qkv", 4, 1024, 1600, 4800, "f32")]),
}


def make_inputs(layer: Layer, seed: int = 0) -> dict:
    """Host arrays (storage dtype) for one layer: dout, inp, weight and the
    initial values of dinp, dweight and dbias (dbias is pre-filled with noise
    so that tests can see it being overwritten)."""
    dt, BT, C, OC = layer.dtype, layer.BT, layer.C, layer.OC
    s = lambda key: STREAM[key] + 16 * layer.layer  # noqa: E731
    out = {}
    out["inp"] = normal((BT, C), dt, seed, s("inp"), 0.0, layer.inp_std)
    out["weight"] = normal((OC, C), dt, seed, s("weight"), 0.0, layer.w_std)
    if layer.dout_kind == "lmhead":
        out["dout"] = lmhead_dout(BT, OC, dt, seed, s("dout"), s("lm_index"), layer.dout_std,
                                  -1.0 / BT)
    else:
        out["dout"] = normal((BT, OC), dt, seed, s("dout"), 0.0, layer.dout_std)
    if layer.init_std > 0:
        out["dinp"] = normal((BT, C), dt, seed, s("dinp_init"), 0.0, layer.init_std)
        out["dweight"] = normal((OC, C), dt, seed, s("dweight_init"), 0.0, layer.init_std)
    else:
        out["dinp"] = np.zeros((BT, C), dtype=_NP[_DT[dt]])
        out["dweight"] = np.zeros((OC, C), dtype=_NP[_DT[dt]])
    out["dbias"] = normal((OC,), dt, seed, s("dbias_init"), 0.0, 1.0)
    return out


# ---------------------------------------------------------------------------
# LayerNorm backward workloads (llm.c dev/cuda/layernorm_backward.cu: B=8, T=1024,
# C=1600 in its main; C=768 is GPT-2 small's width)
# ---------------------------------------------------------------------------

# Stream ids of the LayerNorm inputs (disjoint from the linear layers' ids).
LN_STREAM = {"inp_z": 257, "inp_shift": 258, "inp_scale": 259, "weight": 260, "dout": 261,
             "dinp_init": 262, "dweight_init": 263, "dbias_init": 264}


@dataclass(frozen=True)
class LNProblem:
    """One LayerNorm backward problem: inp, dout, dinp (B,T,C); weight, dweight, dbias (C).

    inp rows are shift + scale * N(0,1) with a per-row shift ~ N(0, 0.5) and a
    per-row scale exp(N(0, 0.5)), so that the row statistics differ from row
    to row; weight ~ N(1, 0.1) (GPT-2 initialises it to one); dout ~ N(0, 1e-2)
    like the gradients the linear layers produce; dinp, dweight and dbias start
    from N(0, init_std) noise so that accumulation is visible."""
    name: str
    B: int
    T: int
    C: int
    dtype: str
    dout_std: float = 1e-2
    init_std: float = 1e-2

    @property
    def BT(self) -> int:
        return self.B * self.T

    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def bytes(self) -> int:
        """Algorithmic HBM bytes: dout and inp read, dinp read and written,
        weight read, dweight and dbias read and written, mean and rstd read."""
        s = self.elem_bytes()
        return 4 * self.BT * self.C * s + 5 * self.C * s + 8 * self.BT


LN_WORKLOADS = {
    "ln_tiny": LNProblem("ln_tiny", 2, 48, 72, "f32", dout_std=1.0),
    "ln_gpt2_small": LNProblem("ln_gpt2_small", 8, 1024, 768, "bf16"),
    "ln_xl": LNProblem("ln_xl", 8, 1024, 1600, "bf16"),
    "ln_xl_f32": LNProblem("ln_xl_f32", 8, 1024, 1600, "f32"),
    # rows wider than the fused kernel stages in shared memory (a 12800-wide
    # hidden state, eight times GPT-2 XL's)
    "ln_wide": LNProblem("ln_wide", 4, 1024, 12800, "bf16"),
}


def round_to(a64: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16 bits (RNE) when dtype is bf16."""
    if dtype == "f64":
        return np.ascontiguousarray(a64, dtype=np.float64)
    f = np.ascontiguousarray(a64, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return f
    bits = f.view(np.uint32).astype(np.uint64)
    return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)


def make_ln_inputs(p: LNProblem, seed: int = 0) -> dict:
    """Host arrays (storage dtype) of one LayerNorm backward problem: inp,
    weight, dout and the initial dinp, dweight, dbias. The row statistics
    (mean, rstd) are not drawn here: they are what the forward caches, so the
    caller derives them from ``inp``."""
    dt, BT, C = p.dtype, p.BT, p.C
    z = normal((BT, C), "f64", seed, LN_STREAM["inp_z"])
    shift = normal((BT, 1), "f64", seed, LN_STREAM["inp_shift"], 0.0, 0.5)
    scale = np.exp(normal((BT, 1), "f64", seed, LN_STREAM["inp_scale"], 0.0, 0.5))
    out = {"inp": round_to(shift + scale * z, dt)}
    out["weight"] = normal((C,), dt, seed, LN_STREAM["weight"], 1.0, 0.1)
    out["dout"] = normal((BT, C), dt, seed, LN_STREAM["dout"], 0.0, p.dout_std)
    out["dinp"] = normal((BT, C), dt, seed, LN_STREAM["dinp_init"], 0.0, p.init_std)
    out["dweight"] = normal((C,), dt, seed, LN_STREAM["dweight_init"], 0.0, p.init_std)
    out["dbias"] = normal((C,), dt, seed, LN_STREAM["dbias_init"], 0.0, p.init_std)
    return out


# ---------------------------------------------------------------------------
# Encoder backward workloads (llm.c llmc/encoder.cuh; GPT-2 small: C=768, padded
# vocabulary V=50304, B=8, T=1024)
# ---------------------------------------------------------------------------

ENC_STREAM = {"tokens": 300, "dout": 301, "dwte_init": 302, "dwpe_init": 303}


@dataclass(frozen=True)
class EncProblem:
    """One encoder backward problem: dout (B,T,C), inp (B,T) token ids, dwte
    (V,C), dwpe (T,C). Token ids follow a Zipf law over the first `V_used` ids
    (p(k) ~ 1/(k+1)^s, the rank-frequency shape of text), so a few tokens
    recur hundreds of times and most once or never, as with real batches."""
    name: str
    B: int
    T: int
    C: int
    V: int
    dtype: str
    V_used: int = 50257
    zipf_s: float = 1.1
    dout_std: float = 1e-2
    init_std: float = 1e-2

    @property
    def BT(self) -> int:
        return self.B * self.T

    def bytes(self, distinct_tokens: int | None = None) -> int:
        """Algorithmic HBM bytes: dout read once, the touched dwte rows read and
        written (distinct_tokens rows; without it, the bound min(B*T, V)), dwpe
        read and written, token ids read."""
        s = 4 if self.dtype == "f32" else 2
        u = min(self.BT, self.V) if distinct_tokens is None else distinct_tokens
        return self.BT * self.C * s + 2 * u * self.C * s + 2 * self.T * self.C * s + 4 * self.BT


ENC_WORKLOADS = {
    "enc_tiny": EncProblem("enc_tiny", 2, 64, 72, 97, "f32", V_used=90, dout_std=1.0),
    "enc_gpt2_small": EncProblem("enc_gpt2_small", 8, 1024, 768, 50304, "bf16"),
    "enc_gpt2_small_f32": EncProblem("enc_gpt2_small_f32", 8, 1024, 768, 50304, "f32"),
}


def zipf_tokens(n: int, v_used: int, s: float, seed: int, stream: int) -> np.ndarray:
    """n token ids in [0, v_used) with p(k) proportional to 1/(k+1)^s, by the
    inverse CDF of uniforms from the counter-based generator."""
    w = 1.0 / np.power(np.arange(1, v_used + 1, dtype=np.float64), s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = uniform(n, seed, stream)
    return np.minimum(np.searchsorted(cdf, u, side="right"), v_used - 1).astype(np.int32)


def make_enc_inputs(p: EncProblem, seed: int = 0) -> dict:
    """Host arrays of one encoder backward problem: inp (int32), dout and the
    initial dwte, dwpe (storage dtype)."""
    dt = p.dtype
    return {
        "inp": zipf_tokens(p.BT, min(p.V_used, p.V), p.zipf_s, seed, ENC_STREAM["tokens"]),
        "dout": normal((p.BT, p.C), dt, seed, ENC_STREAM["dout"], 0.0, p.dout_std),
        "dwte": normal((p.V, p.C), dt, seed, ENC_STREAM["dwte_init"], 0.0, p.init_std),
        "dwpe": normal((p.T, p.C), dt, seed, ENC_STREAM["dwpe_init"], 0.0, p.init_std),
    }
