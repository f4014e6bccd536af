"""GB300 MoE expert layer: thin Python binding of the C ABI in ``include/moe.h``.

Every step of the layer runs in the CUDA kernels of ``libmoe.so``; this module only checks
and marshals arguments.  PyTorch provides device memory and streams.  There is no fallback:
if the library is not built, importing a plan raises.

    plan = MoePlan(E=256, k=8, d_model=2048, d_ff=512, n_shared=1)
    plan.set_weights(w_router, None, w_gate, w_up, w_down)    # device tensors
    plan.set_shared(512, ws_gate, ws_up, ws_down)
    plan.allocate_workspace(T_max=8195)
    out = plan.forward(x, n_prefill=2048)                    # x bf16 [T][d] on the GPU
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB as LIB_PATH

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_NOT_READY = 0, 1, 2, 3
MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE, MOE_ERR_TIMEOUT = 4, 5, 6, 7
MOE_W_BF16, MOE_W_MXFP4 = 0, 1
PATHS = {"auto": 0, "simt": 1, "tc": 2}
DEVERR_EXPERT_RANGE, DEVERR_NONFINITE, DEVERR_TIMEOUT, DEVERR_SEGMENT, DEVERR_RANGE = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED = (
    "moe_plan_create", "moe_plan_destroy", "moe_last_error", "moe_plan_set_weights", "moe_plan_set_shared",
    "moe_plan_workspace_bytes", "moe_plan_set_workspace", "moe_plan_set_path", "moe_layer_forward",
    "moe_route", "moe_route_logits", "moe_permute", "moe_experts", "moe_combine",
    "moe_plan_get_device_error", "moe_plan_enable_timing", "moe_plan_timing_report",
    "moe_plan_last_launch_count", "moe_compose_prefill", "moe_permute_static", "moe_selftest_wait_expiry",
    "moe_plan_resolved_path",
)

_lib = None


class PrefillCall(ctypes.Structure):
    """moe_prefill_call: one layer call of a prompt's prefill."""
    _fields_ = [("pos", ctypes.c_int64), ("n", ctypes.c_int32), ("piece", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"moe status {status}: {msg}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libmoe.so (built by ``decode_batches_gb300.build``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m decode_batches_gb300.build` "
                          "(there is no CPU or eager fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, sz, u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
    sig = {
        "moe_plan_create": ([i32, i32, i32, i32, i32, i32], vp),
        "moe_plan_destroy": ([vp], None),
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_plan_set_weights": ([vp] * 9, i32),
        "moe_plan_set_shared": ([vp, i32, vp, vp, vp], i32),
        "moe_plan_workspace_bytes": ([vp, i32], sz),
        "moe_plan_set_workspace": ([vp, vp, sz, i32], i32),
        "moe_plan_set_path": ([vp, i32], i32),
        "moe_layer_forward": ([vp, vp, i32, i32, vp, vp], i32),
        "moe_route": ([vp, vp, i32, vp, vp, vp, vp], i32),
        "moe_route_logits": ([vp, vp, i32, vp, vp, vp], i32),
        "moe_permute": ([vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "moe_experts": ([vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "moe_combine": ([vp, vp, vp, vp, vp, i32, vp, vp], i32),
        "moe_plan_get_device_error": ([vp, u32p], i32),
        "moe_plan_enable_timing": ([vp, i32], i32),
        "moe_plan_timing_report": ([vp, ctypes.c_char_p, sz], sz),
        "moe_plan_last_launch_count": ([vp], i32),
        "moe_plan_resolved_path": ([vp], i32),
        "moe_compose_prefill": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.POINTER(PrefillCall), ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def compose_prefill(start_pos: int, n_tokens: int, quantum: int, generation_active: bool,
                    prefill_cap: int = 4096):
    """The layer calls that prefill ``n_tokens`` prompt tokens from context position
    ``start_pos`` (moe_compose_prefill): a list of (pos, n, piece) tuples, in order."""
    lib = load_library()
    total = ctypes.c_int64(0)
    _check(lib.moe_compose_prefill(start_pos, n_tokens, quantum, int(bool(generation_active)), prefill_cap, None, 0,
                                   ctypes.byref(total)))
    arr = (PrefillCall * max(1, total.value))()
    _check(lib.moe_compose_prefill(start_pos, n_tokens, quantum, int(bool(generation_active)), prefill_cap, arr,
                                   total.value, ctypes.byref(total)))
    return [(c.pos, c.n, c.piece) for c in arr[:total.value]]


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, load_library().moe_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class MoePlan:
    """One MoE layer plan (C ABI ``moe_plan``)."""

    def __init__(self, E: int, k: int, d_model: int, d_ff: int, n_shared: int = 0, weight_dtype: str = "bf16"):
        self.lib = load_library()
        wd = {"bf16": MOE_W_BF16, "mxfp4": MOE_W_MXFP4}[weight_dtype]
        self.E, self.k, self.d, self.f, self.n_shared, self.weight_dtype = E, k, d_model, d_ff, n_shared, weight_dtype
        self.f_s = 0
        h = self.lib.moe_plan_create(E, k, d_model, d_ff, n_shared, wd)
        if not h:
            raise MoeError(MOE_ERR_INVALID_ARG, self.lib.moe_last_error().decode())
        self._h = ctypes.c_void_p(h)
        self._ws = None
        self.T_max = 0

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self.lib.moe_plan_destroy(h)
            self._h = None

    close = __del__

    # ---- set-up -------------------------------------------------------------------------------
    def set_weights(self, w_router, b_router, w_gate, w_up, w_down, s_gate=None, s_up=None, s_down=None):
        E, d, f = self.E, self.d, self.f
        args = [_dev(w_router, "w_router", torch.float32, (E, d)),
                _dev(b_router, "b_router", torch.float32, (E,))]
        if self.weight_dtype == "bf16":
            args += [_dev(w_gate, "w_gate", torch.bfloat16, (E, f, d)), _dev(w_up, "w_up", torch.bfloat16, (E, f, d)),
                     _dev(w_down, "w_down", torch.bfloat16, (E, d, f)), None, None, None]
        else:
            args += [_dev(w_gate, "w_gate", torch.uint8, (E, f, d // 2)), _dev(w_up, "w_up", torch.uint8, (E, f, d // 2)),
                     _dev(w_down, "w_down", torch.uint8, (E, d, f // 2)),
                     _dev(s_gate, "s_gate", torch.uint8, (E, f, d // 32)), _dev(s_up, "s_up", torch.uint8, (E, f, d // 32)),
                     _dev(s_down, "s_down", torch.uint8, (E, d, f // 32))]
        _check(self.lib.moe_plan_set_weights(self._h, *args))

    def set_shared(self, d_ff_shared: int, w_gate, w_up, w_down):
        n, d, fs = self.n_shared, self.d, d_ff_shared
        _check(self.lib.moe_plan_set_shared(self._h, fs, _dev(w_gate, "w_gate", torch.bfloat16, (n, fs, d)),
                                            _dev(w_up, "w_up", torch.bfloat16, (n, fs, d)),
                                            _dev(w_down, "w_down", torch.bfloat16, (n, d, fs))))
        self.f_s = fs

    def workspace_bytes(self, T_max: int) -> int:
        return int(self.lib.moe_plan_workspace_bytes(self._h, T_max))

    def set_workspace(self, buf: torch.Tensor, T_max: int):
        _check(self.lib.moe_plan_set_workspace(self._h, _dev(buf, "workspace"), buf.numel() * buf.element_size(), T_max))
        self._ws = buf
        self.T_max = T_max

    def allocate_workspace(self, T_max: int, device=None) -> torch.Tensor:
        buf = torch.empty(self.workspace_bytes(T_max), dtype=torch.uint8, device=device or "cuda")
        self.set_workspace(buf, T_max)
        return buf

    def set_path(self, path: str):
        _check(self.lib.moe_plan_set_path(self._h, PATHS[path]))

    # ---- step ---------------------------------------------------------------------------------
    def forward(self, x: torch.Tensor, n_prefill: int = 0, out: Optional[torch.Tensor] = None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.bfloat16, device=x.device)
        _check(self.lib.moe_layer_forward(self._h, _dev(x, "x", torch.bfloat16, (T, self.d)), T, n_prefill,
                                          _dev(out, "out", torch.bfloat16, (T, self.d)), _stream(stream)))
        return out

    def route(self, x: torch.Tensor, want_logits: bool = True, stream=None):
        T = x.shape[0]
        dev = x.device
        logits = torch.empty((T, self.E), dtype=torch.float32, device=dev) if want_logits else None
        ids = torch.empty((T, self.k), dtype=torch.int32, device=dev)
        gates = torch.empty((T, self.k), dtype=torch.float32, device=dev)
        _check(self.lib.moe_route(self._h, _dev(x, "x", torch.bfloat16, (T, self.d)), T, _ptr(logits), _ptr(ids),
                                  _ptr(gates), _stream(stream)))
        return logits, ids, gates

    def route_logits(self, logits: torch.Tensor, stream=None):
        T = logits.shape[0]
        ids = torch.empty((T, self.k), dtype=torch.int32, device=logits.device)
        gates = torch.empty((T, self.k), dtype=torch.float32, device=logits.device)
        _check(self.lib.moe_route_logits(self._h, _dev(logits, "logits", torch.float32, (T, self.E)), T, _ptr(ids),
                                         _ptr(gates), _stream(stream)))
        return ids, gates

    def permute(self, ids: torch.Tensor, stream=None):
        T = ids.shape[0]
        dev = ids.device
        counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        perm = torch.full((T * self.k,), -1, dtype=torch.int32, device=dev)
        inv = torch.empty(T * self.k, dtype=torch.int32, device=dev)
        _check(self.lib.moe_permute(self._h, _dev(ids, "ids", torch.int32, (T, self.k)), T, _ptr(counts), _ptr(offsets),
                                    _ptr(perm), _ptr(inv), _stream(stream)))
        return counts, offsets, perm, inv

    def experts(self, x: torch.Tensor, offsets: torch.Tensor, perm: torch.Tensor, stream=None):
        T = x.shape[0]
        y = torch.empty((T * self.k, self.d), dtype=torch.float16, device=x.device)
        ys = torch.empty((T, self.d), dtype=torch.float16, device=x.device) if self.n_shared else None
        _check(self.lib.moe_experts(self._h, _dev(x, "x", torch.bfloat16, (T, self.d)), T,
                                    _dev(offsets, "offsets", torch.int32, (self.E + 1,)),
                                    _dev(perm, "perm", torch.int32, (T * self.k,)), _ptr(y), _ptr(ys), _stream(stream)))
        return y, ys

    def combine(self, y: torch.Tensor, gates: torch.Tensor, inv: torch.Tensor, shared_y: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, stream=None):
        T = gates.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=torch.bfloat16, device=y.device)
        _check(self.lib.moe_combine(self._h, _dev(y, "y", torch.float32, (T * self.k, self.d)),
                                    _dev(gates, "gates", torch.float32, (T, self.k)),
                                    _dev(inv, "inv", torch.int32, (T * self.k,)),
                                    _dev(shared_y, "shared_y", torch.float32, (T, self.d)), T,
                                    _dev(out, "out", torch.bfloat16, (T, self.d)), _stream(stream)))
        return out

    # ---- diagnostics ----------------------------------------------------------------------------
    def device_error(self) -> int:
        code = ctypes.c_uint32(0)
        st = self.lib.moe_plan_get_device_error(self._h, ctypes.byref(code))
        if st not in (MOE_OK, MOE_ERR_DEVICE):
            _check(st)
        return int(code.value)

    def enable_timing(self, on: bool = True):
        _check(self.lib.moe_plan_enable_timing(self._h, 1 if on else 0))

    def timing_report(self) -> dict:
        """{kernel name: (launches, total ms)} since the last report; synchronises."""
        buf = ctypes.create_string_buffer(1 << 16)
        self.lib.moe_plan_timing_report(self._h, buf, len(buf))
        rep = {}
        for line in buf.value.decode().splitlines():
            name, n, ms = line.split()
            rep[name] = (int(n), float(ms))
        return rep

    def resolved_path(self) -> tuple:
        """('tc' or 'simt', reason): the kernels the expert FFN runs on for this plan."""
        code = int(self.lib.moe_plan_resolved_path(self._h))
        name = {v: k for k, v in PATHS.items()}.get(code, "?")
        return name, ("" if name == "tc" else self.lib.moe_last_error().decode())

    def last_launch_count(self) -> int:
        return int(self.lib.moe_plan_last_launch_count(self._h))
