"""Seeded synthetic inputs for the MoE layer (shared by the oracle's tests and the GPU path).

This package draws numbers and lays them out; it holds none of the layer's arithmetic.
The stream is counter-based (see ``gen.c``), so any slice of any tensor -- one expert's
weights, one token's row -- can be produced on its own and equals the same slice of the
full tensor.

Workloads follow the shapes of the serving steps on the pages (DeepSeek-V4-Flash-like and
Qwen-A3B-like MoE layers; "moe-prefill-quantum", Table 9 and the quantum formula;
"M3 Ultra DSpark" post, the 6-row verify):

* ``tiny``      T=16,  d=256,  E=8,   k=2, f=512,  no shared expert, bf16
* ``decode``    T=4,   d=2048, E=256, k=8, f=512,  one shared expert f_s=512, bf16
* ``mixed``     T=quantum+3 (3 decode rows last), the ``decode`` layer
* ``fp4_zipf``  T=2048+3, d=4096, E=384, k=8, f=1024, shared f_s=2048; routed weights in the
                block-scaled 4-bit format; router bias b[e] = -1.1 ln(e+1) (Zipf s=1.1 prior)
* ``verify``    8 sequences x 6 rows on the ``fp4_zipf`` layer; row = x_seq + 0.1 N(0,1)

Distributions: x ~ N(0,1) rounded to bf16; router weight ~ N(0, 0.02^2) fp32; expert weights
~ N(0, 1/fan_in) (fan_in = d for gate/up, f or f_s for down).  Tensor ids: x=1, router=2,
gate=3, up=4, down=5, shared gate/up/down=6/7/8, sequence rows=9, verify noise=10.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

TID_X, TID_ROUTER, TID_GATE, TID_UP, TID_DOWN = 1, 2, 3, 4, 5
TID_SH_GATE, TID_SH_UP, TID_SH_DOWN, TID_SEQ, TID_NOISE = 6, 7, 8, 9, 10


def build_lib(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_build/libsynth.so`` (gcc, plain C, no arch flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                           "-std=c11", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_lib())
            u64, u32, dbl, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p
            for name in ("synth_normal_f64", "synth_normal_f32", "synth_normal_bf16"):
                getattr(lib, name).argtypes = [u64, u32, u64, u64, dbl, dbl, vp]
                getattr(lib, name).restype = None
            lib.synth_mxfp4.argtypes = [u64, u32, u64, u64, dbl, vp, vp]
            lib.synth_mxfp4.restype = None
            lib.synth_round_bf16.argtypes = [vp, u64, vp]
            lib.synth_round_bf16.restype = None
            lib.synth_set_threads.argtypes = [ctypes.c_int]
            lib.synth_set_threads.restype = None
            lib.synth_set_threads(min(64, os.cpu_count() or 8))
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal_f64(seed: int, tid: int, start: int, count: int, mean: float = 0.0, std: float = 1.0):
    out = np.empty(count, np.float64)
    _load().synth_normal_f64(seed, tid, start, count, mean, std, _ptr(out))
    return out


def normal_f32(seed: int, tid: int, start: int, count: int, mean: float = 0.0, std: float = 1.0):
    out = np.empty(count, np.float32)
    _load().synth_normal_f32(seed, tid, start, count, mean, std, _ptr(out))
    return out


def normal_bf16(seed: int, tid: int, start: int, count: int, mean: float = 0.0, std: float = 1.0):
    """bf16 bit patterns (uint16) of mean + std * z."""
    out = np.empty(count, np.uint16)
    _load().synth_normal_bf16(seed, tid, start, count, mean, std, _ptr(out))
    return out


def mxfp4_blocks(seed: int, tid: int, start_block: int, nblocks: int, std: float):
    """(codes uint8 [nblocks*16], scales uint8 [nblocks]) for N(0, std^2) weights."""
    codes = np.empty(nblocks * 16, np.uint8)
    scales = np.empty(nblocks, np.uint8)
    _load().synth_mxfp4(seed, tid, start_block, nblocks, std, _ptr(codes), _ptr(scales))
    return codes, scales


def round_bf16(values: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint16)
    _load().synth_round_bf16(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(values))


# --------------------------------------------------------------------------------------
# Layer shapes and workloads
# --------------------------------------------------------------------------------------

@dataclass(frozen=True)
class LayerSpec:
    E: int            # routed experts
    k: int            # experts per token
    d: int            # d_model
    f: int            # d_ff of a routed expert
    n_shared: int     # always-on shared experts (weight 1 each)
    f_s: int          # d_ff of a shared expert
    wdtype: str       # "bf16" or "mxfp4" (routed experts; shared experts are always bf16)
    zipf_s: Optional[float] = None  # router bias b[e] = -s ln(e+1), else zero bias


@dataclass
class ExpertWeights:
    """Routed expert weights as stored for the GPU (bf16 bits or 4-bit codes + scales)."""
    spec: LayerSpec
    gate: np.ndarray                 # bf16: uint16 [E][f][d]; mxfp4: uint8 [E][f][d/2]
    up: np.ndarray
    down: np.ndarray                 # bf16: uint16 [E][d][f]; mxfp4: uint8 [E][d][f/2]
    gate_scale: Optional[np.ndarray] = None  # uint8 [E][f][d/32]
    up_scale: Optional[np.ndarray] = None
    down_scale: Optional[np.ndarray] = None  # uint8 [E][d][f/32]


@dataclass
class Workload:
    name: str
    spec: LayerSpec
    T: int
    n_prefill: int
    seed: int = 0
    x_kind: str = "normal"        # "normal" or "verify"
    verify_seqs: int = 0
    verify_rows: int = 0
    _cache: dict = field(default_factory=dict, repr=False)

    # ---- activations -------------------------------------------------------------
    def x(self) -> np.ndarray:
        """bf16 bits uint16 [T][d]."""
        if "x" not in self._cache:
            d = self.spec.d
            if self.x_kind == "normal":
                xs = normal_bf16(self.seed, TID_X, 0, self.T * d)
            else:
                seq = normal_f64(self.seed, TID_SEQ, 0, self.verify_seqs * d).reshape(self.verify_seqs, d)
                noise = normal_f64(self.seed, TID_NOISE, 0, self.T * d).reshape(self.T, d)
                rows = np.repeat(seq, self.verify_rows, axis=0) + 0.1 * noise
                xs = round_bf16(rows)
            self._cache["x"] = xs.reshape(self.T, d)
        return self._cache["x"]

    # ---- router --------------------------------------------------------------------
    def router_weight(self) -> np.ndarray:
        """fp32 [E][d], N(0, 0.02^2)."""
        if "wr" not in self._cache:
            s = self.spec
            self._cache["wr"] = normal_f32(self.seed, TID_ROUTER, 0, s.E * s.d, 0.0, 0.02).reshape(s.E, s.d)
        return self._cache["wr"]

    def router_bias(self) -> Optional[np.ndarray]:
        """fp32 [E] or None.  Zipf(s) popularity prior: b[e] = -s ln(e + 1)."""
        s = self.spec
        if s.zipf_s is None:
            return None
        return np.array([-s.zipf_s * math.log(e + 1.0) for e in range(s.E)], dtype=np.float32)

    # ---- routed experts ----------------------------------------------------------
    def expert_slice(self, e0: int, e1: int) -> ExpertWeights:
        """Weights of experts [e0, e1) (slices of the full tensors, generated on their own)."""
        s = self.spec
        n = e1 - e0
        sg, sd = 1.0 / math.sqrt(s.d), 1.0 / math.sqrt(s.f)
        if s.wdtype == "bf16":
            g = normal_bf16(self.seed, TID_GATE, e0 * s.f * s.d, n * s.f * s.d, 0.0, sg)
            u = normal_bf16(self.seed, TID_UP, e0 * s.f * s.d, n * s.f * s.d, 0.0, sg)
            dn = normal_bf16(self.seed, TID_DOWN, e0 * s.d * s.f, n * s.d * s.f, 0.0, sd)
            return ExpertWeights(s, g.reshape(n, s.f, s.d), u.reshape(n, s.f, s.d), dn.reshape(n, s.d, s.f))
        assert s.wdtype == "mxfp4" and s.d % 32 == 0 and s.f % 32 == 0
        bg = s.f * s.d // 32
        bd = s.d * s.f // 32
        gc, gs = mxfp4_blocks(self.seed, TID_GATE, e0 * bg, n * bg, sg)
        uc, us = mxfp4_blocks(self.seed, TID_UP, e0 * bg, n * bg, sg)
        dc, ds = mxfp4_blocks(self.seed, TID_DOWN, e0 * bd, n * bd, sd)
        return ExpertWeights(
            s, gc.reshape(n, s.f, s.d // 2), uc.reshape(n, s.f, s.d // 2), dc.reshape(n, s.d, s.f // 2),
            gs.reshape(n, s.f, s.d // 32), us.reshape(n, s.f, s.d // 32), ds.reshape(n, s.d, s.f // 32))

    def experts(self) -> ExpertWeights:
        if "experts" not in self._cache:
            self._cache["experts"] = self.expert_slice(0, self.spec.E)
        return self._cache["experts"]

    # ---- shared experts (bf16) ---------------------------------------------------------
    def shared(self):
        """(gate [n_s][f_s][d], up [n_s][f_s][d], down [n_s][d][f_s]) bf16 bits, or None."""
        s = self.spec
        if s.n_shared == 0:
            return None
        if "shared" not in self._cache:
            n = s.n_shared * s.f_s * s.d
            sg, sd = 1.0 / math.sqrt(s.d), 1.0 / math.sqrt(s.f_s)
            g = normal_bf16(self.seed, TID_SH_GATE, 0, n, 0.0, sg).reshape(s.n_shared, s.f_s, s.d)
            u = normal_bf16(self.seed, TID_SH_UP, 0, n, 0.0, sg).reshape(s.n_shared, s.f_s, s.d)
            dn = normal_bf16(self.seed, TID_SH_DOWN, 0, n, 0.0, sd).reshape(s.n_shared, s.d, s.f_s)
            self._cache["shared"] = (g, u, dn)
        return self._cache["shared"]

    def drop_cache(self):
        self._cache.clear()


TINY = LayerSpec(E=8, k=2, d=256, f=512, n_shared=0, f_s=0, wdtype="bf16")
QWEN_A3B_LIKE = LayerSpec(E=256, k=8, d=2048, f=512, n_shared=1, f_s=512, wdtype="bf16")
FP4_ZIPF = LayerSpec(E=384, k=8, d=4096, f=1024, n_shared=1, f_s=2048, wdtype="mxfp4", zipf_s=1.1)

QUANTA = (128, 512, 1024, 2048, 4096, 8192)


def workload(name: str, quantum: int = 2048, seed: int = 0) -> Workload:
    """Named workloads; ``mixed`` takes the prefill quantum (T = quantum + 3 decode rows)."""
    if name == "tiny":
        return Workload("tiny", TINY, T=16, n_prefill=16, seed=seed)
    if name == "decode":
        return Workload("decode", QWEN_A3B_LIKE, T=4, n_prefill=0, seed=seed)
    if name == "mixed":
        return Workload(f"mixed_q{quantum}", QWEN_A3B_LIKE, T=quantum + 3, n_prefill=quantum, seed=seed)
    if name == "fp4_zipf":
        return Workload("fp4_zipf", FP4_ZIPF, T=2048 + 3, n_prefill=2048, seed=seed)
    if name == "verify":
        return Workload("verify", FP4_ZIPF, T=48, n_prefill=0, seed=seed, x_kind="verify",
                        verify_seqs=8, verify_rows=6)
    raise KeyError(name)


def custom(spec: LayerSpec, T: int, n_prefill: int = 0, seed: int = 0, name: str = "custom") -> Workload:
    return Workload(name, spec, T=T, n_prefill=n_prefill, seed=seed)
