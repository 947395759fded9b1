"""ctypes binding of librssm.so: argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels. This module
checks tensor shapes, dtypes and devices, allocates the caller-owned workspace
with PyTorch (which provides device memory and streams), and passes raw
pointers through the C ABI declared in ``include/rssm.h``. No computation of
the method happens here. No CPU fallback exists: if the library is missing,
the import raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# The in-tree build (hybrid_model_ssm_gb300.build).
LIB_PATH = os.path.join(_HERE, "librssm.so")

RSSM_OK, RSSM_EINVAL, RSSM_ECAPACITY, RSSM_ECUDA, RSSM_EUNSUPPORTED, RSSM_ETIMEOUT = range(6)
STATUS_NAMES = {0: "RSSM_OK", 1: "RSSM_EINVAL", 2: "RSSM_ECAPACITY", 3: "RSSM_ECUDA", 4: "RSSM_EUNSUPPORTED",
                5: "RSSM_ETIMEOUT"}
DTYPES = {"f32": 0, "bf16": 1}
READ_FMTS = {None: 0, "none": 0, "e4m3": 1, "e2m1": 2}
CKPT_FMTS = {"f32": 0, "f16_sr": 1, "f16_rn": 2}
RECURRENCES = {"outer": 0, "delta": 1}
ERR_CAPACITY, ERR_ACCEPT, ERR_TIMEOUT, ERR_PLAN = 1, 2, 4, 8

# The C ABI functions, with their argument types.
_c_size_p = ctypes.POINTER(ctypes.c_size_t)
_c_i32_p = ctypes.POINTER(ctypes.c_int32)
_c_u32_p = ctypes.POINTER(ctypes.c_uint32)
_vp = ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "H", "P", "N", "G", "L", "T_max", "in_dtype", "read_fmt",
                                              "ckpt_fmt")] + [("seed", ctypes.c_uint64), ("recurrence", ctypes.c_int32)]


class LaunchPlanInfo(ctypes.Structure):
    _fields_ = [("smem_bytes", ctypes.c_int64), ("nonflush_layout", ctypes.c_int32)] + [
        (n, ctypes.c_int32 * 2) for n in ("stages", "stage_bytes", "slots", "slot_bytes", "dgroups")]


_Cfg_p = ctypes.POINTER(Config)
SIGNATURES = {
    "rssm_workspace_size": [_Cfg_p, _c_size_p, _c_size_p, _c_size_p],
    "rssm_ring_offsets": [_Cfg_p, _c_size_p, _c_size_p],
    "rssm_read_copy_layout": [_Cfg_p, _c_size_p, _c_size_p, _c_size_p],
    "rssm_launch_plan": [_Cfg_p, ctypes.c_int32, ctypes.POINTER(LaunchPlanInfo)],
    "rssm_create": [_Cfg_p, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)],
    "rssm_decode_step": [_vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_decode_step_static_scratch": [_vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_decode_step_delta": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_verify": [_vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_verify_delta": [_vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_set_decode_kernel": [_vp, ctypes.c_int32],
    "rssm_get_decode_kernel": [_vp, _c_i32_p],
    "rssm_set_verify_kernel": [_vp, ctypes.c_int32],
    "rssm_get_verify_kernel": [_vp, ctypes.c_int32, _c_i32_p],
    "rssm_commit": [_vp, _vp, _vp],
    "rssm_flush": [_vp, ctypes.c_int32, _vp],
    "rssm_read_pointers": [_vp, _c_i32_p, _c_i32_p, _c_u32_p, _vp],
    "rssm_clear_error": [_vp, _vp],
    "rssm_selftest_bounded_wait": [_vp, _vp],
    "rssm_destroy": [_vp],
    "rssm_last_error": [],
    "rssm_conventional_step": [_Cfg_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_conventional_step_delta": [_Cfg_p, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_conventional_verify": [_Cfg_p, _vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "rssm_conventional_commit": [_Cfg_p, _vp, _vp, ctypes.c_int32, _vp, _vp],
    "rssm_round_f16": [_vp, _vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32, _vp],
}


class RssmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load librssm.so. Raises if it has not been built (no fallback exists)."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m hybrid_model_ssm_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "rssm_last_error" else ctypes.c_int
    return lib


_LIB: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def _check(status: int):
    if status != RSSM_OK:
        raise RssmError(status, lib().rssm_last_error().decode())


@dataclass(frozen=True)
class LayerShape:
    """Sizes of one SSM layer (see include/rssm.h for their meaning)."""

    B: int
    H: int
    P: int
    N: int
    G: int
    L: int
    T_max: int = 1
    in_dtype: str = "bf16"
    read_fmt: str | None = None
    ckpt: str = "f32"  # checkpoint storage: "f32", "f16_sr" (stochastic rounding) or "f16_rn"
    seed: int = 0      # key of the stochastic rounding
    recurrence: str = "outer"  # "outer" (gated outer product) or "delta" (gated delta rule)

    @property
    def R(self) -> int:
        return self.L + self.T_max - 1

    @property
    def torch_in_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "f32": torch.float32}[self.in_dtype]

    @property
    def torch_ckpt_dtype(self) -> torch.dtype:
        return torch.float32 if self.ckpt == "f32" else torch.float16

    def config(self) -> Config:
        return Config(self.B, self.H, self.P, self.N, self.G, self.L, self.T_max, DTYPES[self.in_dtype],
                      READ_FMTS[self.read_fmt], CKPT_FMTS[self.ckpt], self.seed, RECURRENCES[self.recurrence])


def workspace_size(shape: LayerShape) -> tuple[int, int, int]:
    c = shape.config()
    r, p, q = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().rssm_workspace_size(ctypes.byref(c), ctypes.byref(r), ctypes.byref(p), ctypes.byref(q)))
    return r.value, p.value, q.value


def ring_offsets(shape: LayerShape) -> tuple[int, int]:
    c = shape.config()
    v, k = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().rssm_ring_offsets(ctypes.byref(c), ctypes.byref(v), ctypes.byref(k)))
    return v.value, k.value


def read_copy_layout(shape: LayerShape) -> tuple[int, int, int]:
    c = shape.config()
    a, b, d = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().rssm_read_copy_layout(ctypes.byref(c), ctypes.byref(a), ctypes.byref(b), ctypes.byref(d)))
    return a.value, b.value, d.value


LAUNCH_KINDS = {"flush": 0, "decode": 1, "verify": 2, "verify_tc": 3, "warp_per_head": 4}
VERIFY_KERNELS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2}
DECODE_KERNELS = {"auto": 0, "head_kernel": 1, "warp_per_head": 2}


def launch_plan(shape: LayerShape, kind: str) -> dict:
    """Shared-memory plan of a launch kind ("flush", "decode", "verify", "verify_tc",
    "warp_per_head"): smem bytes and, per layout, stages, stage bytes, slots, slot bytes and
    dot-warp groups (for "warp_per_head": two tile stages and one value stage per warp, and
    the warps per CTA in dgroups)."""
    c = shape.config()
    info = LaunchPlanInfo()
    _check(lib().rssm_launch_plan(ctypes.byref(c), LAUNCH_KINDS[kind], ctypes.byref(info)))
    layouts = 2 if kind == "decode" and info.nonflush_layout else 1
    return {"smem_bytes": info.smem_bytes,
            "layouts": [{f: getattr(info, f)[i] for f in ("stages", "stage_bytes", "slots", "slot_bytes", "dgroups")}
                        for i in range(layouts)]}


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _expect(t: torch.Tensor, shape, dtype, name: str, device: torch.device | None = None):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, the layer's state is on {device}")


class ReplaySSM:
    """One SSM layer's replay decoding state, bound to caller (PyTorch) memory.

    ``ckpt`` [B,H,P,N] fp32 on the GPU is the initial state. It is updated in
    place at every flush. The ring, the pointer block and the optional read copy
    are allocated here as plain uint8 CUDA tensors and then belong to this object.
    """

    def __init__(self, shape: LayerShape, ckpt: torch.Tensor, stream=None):
        _expect(ckpt, (shape.B, shape.H, shape.P, shape.N), shape.torch_ckpt_dtype, "ckpt")
        self.shape = shape
        self.ckpt = ckpt
        ring_b, ptr_b, copy_b = workspace_size(shape)
        dev = ckpt.device
        self.ring = torch.empty(ring_b, dtype=torch.uint8, device=dev)
        self.ptrs = torch.empty(ptr_b, dtype=torch.uint8, device=dev)
        self.copy = torch.empty(copy_b, dtype=torch.uint8, device=dev) if copy_b else None
        self._cfg = shape.config()
        self._dev_index = dev.index if dev.index is not None else torch.cuda.current_device()
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _check(lib().rssm_create(ctypes.byref(self._cfg), _ptr(ckpt), _ptr(self.ring), _ptr(self.ptrs),
                                     _ptr(self.copy), _stream_ptr(stream), ctypes.byref(h)))
        self._h = h

    def _on_device(self):
        """The layer's device made current for a call (nothing to do when it already is)."""
        if torch.cuda.current_device() == self._dev_index:
            return contextlib.nullcontext()
        return torch.cuda.device(self._dev_index)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _LIB is not None:
            _LIB.rssm_destroy(h)
            self._h = None

    # ------------------------------------------------------------ decode path
    def decode_step(self, alpha, v, k, q, out=None, stream=None, beta=None) -> torch.Tensor:
        """One decode step; a delta-rule layer also takes beta [B,H] fp32."""
        s, d = self.shape, self.ckpt.device
        _expect(alpha, (s.B, s.H), torch.float32, "alpha", d)
        if (beta is None) != (s.recurrence == "outer"):
            raise ValueError("beta is required for (and only for) a delta-rule layer")
        _expect(v, (s.B, s.H, s.P), s.torch_in_dtype, "v", d)
        _expect(k, (s.B, s.G, s.N), s.torch_in_dtype, "k", d)
        _expect(q, (s.B, s.G, s.N), s.torch_in_dtype, "q", d)
        if out is None:
            out = torch.empty((s.B, s.H, s.P), dtype=torch.float32, device=d)
        _expect(out, (s.B, s.H, s.P), torch.float32, "out", d)
        with self._on_device():
            if beta is None:
                _check(lib().rssm_decode_step(self._h, _ptr(alpha), _ptr(v), _ptr(k), _ptr(q), _ptr(out),
                                              _stream_ptr(stream)))
            else:
                _expect(beta, (s.B, s.H), torch.float32, "beta", d)
                _check(lib().rssm_decode_step_delta(self._h, _ptr(alpha), _ptr(beta), _ptr(v), _ptr(k), _ptr(q),
                                                    _ptr(out), _stream_ptr(stream)))
        return out

    def decode_step_static_scratch(self, alpha, v, k, q, out=None, stream=None) -> torch.Tensor:
        """One decode step of an outer-product layer with its tickets in the library's
        static device array instead of the pointer block (B <= 8192)."""
        s, d = self.shape, self.ckpt.device
        _expect(alpha, (s.B, s.H), torch.float32, "alpha", d)
        _expect(v, (s.B, s.H, s.P), s.torch_in_dtype, "v", d)
        _expect(k, (s.B, s.G, s.N), s.torch_in_dtype, "k", d)
        _expect(q, (s.B, s.G, s.N), s.torch_in_dtype, "q", d)
        if out is None:
            out = torch.empty((s.B, s.H, s.P), dtype=torch.float32, device=d)
        _expect(out, (s.B, s.H, s.P), torch.float32, "out", d)
        with self._on_device():
            _check(lib().rssm_decode_step_static_scratch(self._h, _ptr(alpha), _ptr(v), _ptr(k), _ptr(q),
                                                         _ptr(out), _stream_ptr(stream)))
        return out

    def verify(self, alpha, v, k, q, out=None, stream=None, beta=None) -> torch.Tensor:
        """Speculative verify of T drafts; a delta-rule layer also takes beta [B,T,H] fp32."""
        s, d = self.shape, self.ckpt.device
        T = alpha.shape[1]
        if (beta is None) != (s.recurrence == "outer"):
            raise ValueError("beta is required for (and only for) a delta-rule layer")
        _expect(alpha, (s.B, T, s.H), torch.float32, "alpha", d)
        _expect(v, (s.B, T, s.H, s.P), s.torch_in_dtype, "v", d)
        _expect(k, (s.B, T, s.G, s.N), s.torch_in_dtype, "k", d)
        _expect(q, (s.B, T, s.G, s.N), s.torch_in_dtype, "q", d)
        if out is None:
            out = torch.empty((s.B, T, s.H, s.P), dtype=torch.float32, device=d)
        _expect(out, (s.B, T, s.H, s.P), torch.float32, "out", d)
        with torch.cuda.device(d):
            if beta is None:
                _check(lib().rssm_verify(self._h, T, _ptr(alpha), _ptr(v), _ptr(k), _ptr(q), _ptr(out),
                                         _stream_ptr(stream)))
            else:
                _expect(beta, (s.B, T, s.H), torch.float32, "beta", d)
                _check(lib().rssm_verify_delta(self._h, T, _ptr(alpha), _ptr(beta), _ptr(v), _ptr(k), _ptr(q),
                                               _ptr(out), _stream_ptr(stream)))
        return out

    def set_decode_kernel(self, kind: str):
        """Kernels of the decode steps: "auto", "head_kernel" (alone) or "warp_per_head"
        (the non-flush step of read copies and FP16 checkpoints, then the head kernel)."""
        _check(lib().rssm_set_decode_kernel(self._h, DECODE_KERNELS[kind]))

    def decode_kernel(self) -> str:
        """The kernels a decode step launches: "head_kernel" or "warp_per_head"."""
        k = ctypes.c_int32()
        _check(lib().rssm_get_decode_kernel(self._h, ctypes.byref(k)))
        return {1: "head_kernel", 2: "warp_per_head"}[k.value]

    def set_verify_kernel(self, kind: str):
        """Kernel of the verify launches: "auto", "cuda_cores" (T <= 8) or "tensor_cores"."""
        _check(lib().rssm_set_verify_kernel(self._h, VERIFY_KERNELS[kind]))

    def verify_kernel(self, T: int) -> str:
        """The kernel a verify of T drafts launches: "cuda_cores" or "tensor_cores"."""
        k = ctypes.c_int32()
        _check(lib().rssm_get_verify_kernel(self._h, int(T), ctypes.byref(k)))
        return {1: "cuda_cores", 2: "tensor_cores"}[k.value]

    def commit(self, accepted: torch.Tensor, stream=None):
        _expect(accepted, (self.shape.B,), torch.int32, "accepted", self.ckpt.device)
        with torch.cuda.device(self.ckpt.device):
            _check(lib().rssm_commit(self._h, _ptr(accepted), _stream_ptr(stream)))

    def flush(self, min_count: int | None = None, stream=None):
        with torch.cuda.device(self.ckpt.device):
            _check(lib().rssm_flush(self._h, self.shape.L if min_count is None else int(min_count),
                                    _stream_ptr(stream)))

    def read_pointers(self, stream=None, check: bool = True):
        """(start, count, error word) as host int32 tensors and an int; synchronizes the stream."""
        B = self.shape.B
        start = (ctypes.c_int32 * B)()
        count = (ctypes.c_int32 * B)()
        err = ctypes.c_uint32()
        with torch.cuda.device(self.ckpt.device):
            st = lib().rssm_read_pointers(self._h, start, count, ctypes.byref(err), _stream_ptr(stream))
        if check:
            _check(st)
        return (torch.tensor(list(start), dtype=torch.int32), torch.tensor(list(count), dtype=torch.int32),
                int(err.value))

    def clear_error(self, stream=None):
        """Zero the device error word and the per-sequence tickets (after a launch that
        gave up on a wait); enqueued on the stream."""
        with torch.cuda.device(self.ckpt.device):
            _check(lib().rssm_clear_error(self._h, _stream_ptr(stream)))

    # ------------------------------------------------------- ring inspection
    def ring_views(self):
        """(alpha [B,H,Rp] f32, V [B,H,R,P], K [B,G,R,N]) views of the ring buffer (for tests).

        V is in the input dtype; a delta-rule layer keeps its pseudo-values there, in f32.
        """
        s = self.shape
        R, Rp = s.R, (s.R + 3) // 4 * 4
        v_off, k_off = ring_offsets(s)
        es = 4 if s.in_dtype == "f32" else 2
        vdt, ves = (torch.float32, 4) if s.recurrence == "delta" else (s.torch_in_dtype, es)
        a = self.ring[: s.B * s.H * Rp * 4].view(torch.float32).view(s.B, s.H, Rp)
        V = self.ring[v_off: v_off + s.B * s.H * R * s.P * ves].view(vdt).view(s.B, s.H, R, s.P)
        K = self.ring[k_off: k_off + s.B * s.G * R * s.N * es].view(s.torch_in_dtype).view(s.B, s.G, R, s.N)
        return a, V, K

    def ring_pseudo_values(self):
        """Pseudo-values w [B,H,R,P] f32 of a delta-rule layer's ring (where V sits for the other recurrence)."""
        s = self.shape
        if s.recurrence != "delta":
            raise ValueError("only delta-rule layers keep pseudo-values")
        return self.ring_views()[1]


def conventional_step(shape: LayerShape, state, alpha, v, k, q, out=None, stream=None, beta=None) -> torch.Tensor:
    """The comparison kernel: S <- alpha S + v k^T, o = S q, state read and written in full.

    For a delta-rule shape (beta [B,H] given): S <- alpha S (I - beta k k^T) + beta v k^T.
    """
    s = shape
    _expect(state, (s.B, s.H, s.P, s.N), torch.float32, "state")
    d = state.device
    _expect(alpha, (s.B, s.H), torch.float32, "alpha", d)
    _expect(v, (s.B, s.H, s.P), s.torch_in_dtype, "v", d)
    _expect(k, (s.B, s.G, s.N), s.torch_in_dtype, "k", d)
    _expect(q, (s.B, s.G, s.N), s.torch_in_dtype, "q", d)
    if out is None:
        out = torch.empty((s.B, s.H, s.P), dtype=torch.float32, device=d)
    _expect(out, (s.B, s.H, s.P), torch.float32, "out", d)
    cfg = s.config()
    with torch.cuda.device(d):
        if beta is None:
            _check(lib().rssm_conventional_step(ctypes.byref(cfg), _ptr(state), _ptr(alpha), _ptr(v), _ptr(k),
                                                _ptr(q), _ptr(out), _stream_ptr(stream)))
        else:
            _expect(beta, (s.B, s.H), torch.float32, "beta", d)
            _check(lib().rssm_conventional_step_delta(ctypes.byref(cfg), _ptr(state), _ptr(alpha), _ptr(beta),
                                                      _ptr(v), _ptr(k), _ptr(q), _ptr(out), _stream_ptr(stream)))
    return out


class ConventionalVerifier:
    """Comparison path: conventional speculative verify with per-draft state snapshots.

    The state of every sequence sits in one of T_max + 1 slots of ``states``
    ([T_max + 1, B, H, P, N] fp32, allocated here; slot 0 starts as ``state0``).
    ``verify`` advances the full state through the T drafts and writes a snapshot
    after each (one state read, T writes); ``commit`` points each sequence at the
    snapshot after its accepted drafts. ``err`` is the device error word.
    """

    def __init__(self, shape: LayerShape, state0: torch.Tensor):
        s = shape
        _expect(state0, (s.B, s.H, s.P, s.N), torch.float32, "state0")
        self.shape = shape
        self.nslot = s.T_max + 1
        self.states = torch.empty((self.nslot, s.B, s.H, s.P, s.N), dtype=torch.float32, device=state0.device)
        self.states[0].copy_(state0)
        self.cur = torch.zeros(s.B, dtype=torch.int32, device=state0.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=state0.device)
        self._cfg = s.config()
        self._last_T = 0

    def verify(self, alpha, v, k, q, out=None, stream=None) -> torch.Tensor:
        s, d = self.shape, self.states.device
        T = alpha.shape[1]
        _expect(alpha, (s.B, T, s.H), torch.float32, "alpha", d)
        _expect(v, (s.B, T, s.H, s.P), s.torch_in_dtype, "v", d)
        _expect(k, (s.B, T, s.G, s.N), s.torch_in_dtype, "k", d)
        _expect(q, (s.B, T, s.G, s.N), s.torch_in_dtype, "q", d)
        if out is None:
            out = torch.empty((s.B, T, s.H, s.P), dtype=torch.float32, device=d)
        _expect(out, (s.B, T, s.H, s.P), torch.float32, "out", d)
        with torch.cuda.device(d):
            _check(lib().rssm_conventional_verify(ctypes.byref(self._cfg), _ptr(self.states), _ptr(self.cur), T,
                                                  _ptr(alpha), _ptr(v), _ptr(k), _ptr(q), _ptr(out), _ptr(self.err),
                                                  _stream_ptr(stream)))
        self._last_T = T
        return out

    def commit(self, accepted: torch.Tensor, stream=None):
        _expect(accepted, (self.shape.B,), torch.int32, "accepted", self.states.device)
        if self._last_T < 1:
            raise ValueError("commit without a pending verify")
        with torch.cuda.device(self.states.device):
            _check(lib().rssm_conventional_commit(ctypes.byref(self._cfg), _ptr(self.cur), _ptr(accepted),
                                                  self._last_T, _ptr(self.err), _stream_ptr(stream)))
        self._last_T = 0

    def state(self) -> torch.Tensor:
        """The committed state [B,H,P,N] (gathered from each sequence's slot; a copy)."""
        idx = self.cur.long()
        return self.states[idx, torch.arange(self.shape.B, device=idx.device)]


def round_f16(x: torch.Tensor, base: int = 0, epoch: int = 0, seed: int = 0, stochastic: bool = True,
              stream=None) -> torch.Tensor:
    """The FP16 checkpoint store's rounding applied to x (fp32, on the GPU); returns fp16 (test support)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    y = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check(lib().rssm_round_f16(_ptr(x), _ptr(y), x.numel(), base, epoch, seed, 1 if stochastic else 0,
                                _stream_ptr(stream)))
    return y
