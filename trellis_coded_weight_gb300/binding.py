"""Thin ctypes binding of libtrellis.so (the C ABI in include/trellis.h).

Argument marshalling only: each function checks the tensors' device, dtype,
shape and contiguity, passes raw device pointers and the current CUDA stream
to the C entry point of the same name, and raises on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback -- if the library cannot be loaded, every call raises.

bf16 tensors are torch.bfloat16; fp16 scales are torch.float16; codes are
torch.int32 or torch.uint32 tensors holding the packed words.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtrellis.so")

TRELLIS_OK = 0
STATUS_NAMES = {0: "TRELLIS_OK", -1: "TRELLIS_EGEOM", -2: "TRELLIS_EM", -3: "TRELLIS_EALIGN", -4: "TRELLIS_EAXIS",
                -5: "TRELLIS_EWORKSPACE", -6: "TRELLIS_ECUDA", -7: "TRELLIS_ENULL", -8: "TRELLIS_EDEVICE"}

EXPORTS = ("trellis_abi_version", "trellis_status_string", "trellis_check_geom", "trellis_expand_bf16",
           "trellis_matvec_axis1", "trellis_matvec_axis0", "trellis_workspace_bytes", "trellis_gateup_swiglu",
           "trellis_gemm_prefill", "trellis_device_error", "trellis_mlp_decode", "trellis_matvec_axis1_bf16w",
           "trellis_matvec_axis0_bf16w", "trellis_load_floor", "trellis_load_floor_rows", "trellis_prefill_plan",
           "trellis_set_wait_limit", "trellis_matvec_axis1_host")


class TrellisGeom(ctypes.Structure):
    """Mirror of trellis_geom_t."""
    _fields_ = [("k", ctypes.c_int32), ("L", ctypes.c_int32), ("T", ctypes.c_int32), ("axis", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("interleave", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


@dataclass(frozen=True)
class Geometry:
    """Stored-matrix geometry: k bits/weight, L-bit windows, T-long blocks."""
    k: int
    L: int
    T: int
    axis: int
    rows: int
    cols: int
    interleave: int = 0  # 2: the k=3 axis-0 layout [cols/512][rows][48]

    def c(self) -> TrellisGeom:
        """The C struct of this geometry (built once per geometry and kept)."""
        g = _GEOM_STRUCTS.get(self)
        if g is None:
            g = _GEOM_STRUCTS.setdefault(self, TrellisGeom(self.k, self.L, self.T, self.axis, self.rows, self.cols,
                                                           self.interleave, 0))
        return g

    @property
    def words_per_row(self) -> int:
        return self.cols * self.k // 32

    @property
    def codes_shape(self) -> tuple:
        if self.interleave:
            return (self.cols // (2 * self.T), self.rows, 2 * self.T * self.k // 32)
        return (self.rows, self.words_per_row)


_GEOM_STRUCTS: dict = {}


class TrellisError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({msg})")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libtrellis.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libtrellis.so not built at {path}; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            g = ctypes.POINTER(TrellisGeom)
            lib.trellis_abi_version.restype = i32
            lib.trellis_abi_version.argtypes = []
            lib.trellis_status_string.restype = ctypes.c_char_p
            lib.trellis_status_string.argtypes = [i32]
            lib.trellis_check_geom.restype = i32
            lib.trellis_check_geom.argtypes = [g]
            lib.trellis_expand_bf16.restype = i32
            lib.trellis_expand_bf16.argtypes = [vp, vp, vp, g, vp]
            lib.trellis_matvec_axis1.restype = i32
            lib.trellis_matvec_axis1.argtypes = [vp, vp, vp, vp, i32, g, vp]
            lib.trellis_matvec_axis0.restype = i32
            lib.trellis_matvec_axis0.argtypes = [vp, vp, vp, vp, i32, g, vp, sz, vp]
            lib.trellis_workspace_bytes.restype = sz
            lib.trellis_workspace_bytes.argtypes = [i32, g]
            lib.trellis_gateup_swiglu.restype = i32
            lib.trellis_gateup_swiglu.argtypes = [vp, vp, vp, vp, vp, vp, i32, g, vp]
            lib.trellis_gemm_prefill.restype = i32
            lib.trellis_gemm_prefill.argtypes = [vp, vp, vp, vp, i32, g, vp]
            lib.trellis_matvec_axis1_host.restype = i32
            lib.trellis_matvec_axis1_host.argtypes = [vp, vp, vp, vp, i32, g, vp, vp, vp]
            lib.trellis_matvec_axis1_bf16w.restype = i32
            lib.trellis_matvec_axis1_bf16w.argtypes = [vp, vp, vp, vp, i32, g, vp]
            lib.trellis_matvec_axis0_bf16w.restype = i32
            lib.trellis_matvec_axis0_bf16w.argtypes = [vp, vp, vp, vp, i32, g, vp, sz, vp]
            lib.trellis_mlp_decode.restype = i32
            lib.trellis_mlp_decode.argtypes = [vp] * 9 + [i32, g, g, vp, sz, vp]
            lib.trellis_device_error.restype = i32
            lib.trellis_device_error.argtypes = [i32]
            lib.trellis_set_wait_limit.restype = i32
            lib.trellis_set_wait_limit.argtypes = [ctypes.c_uint64]
            lib.trellis_load_floor.restype = i32
            lib.trellis_load_floor.argtypes = [vp, vp, g, vp]
            lib.trellis_load_floor_rows.restype = i32
            lib.trellis_load_floor_rows.argtypes = [vp, vp, g, vp]
            lib.trellis_prefill_plan.restype = i32
            lib.trellis_prefill_plan.argtypes = [i32, g, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != TRELLIS_OK:
        raise TrellisError(fn, status, load().trellis_status_string(status).decode())


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _on(t: torch.Tensor):
    """Make the tensor's device current for the C call: the library reads the
    current device (its SM count, kernel attributes) and launches on it."""
    if t.device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def _req(t: torch.Tensor, name: str, dtypes, shape):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_CODES = (torch.int32, getattr(torch, "uint32", torch.int32))


def expand_bf16(codes, scales, g: Geometry, out=None):
    """Decoded stored matrix [rows, cols] bf16 (bit-exact)."""
    if out is None:
        out = torch.empty((g.rows, g.cols), dtype=torch.bfloat16, device=codes.device)
    args = (_req(codes, "codes", _CODES, g.codes_shape),
            _req(scales, "scales", (torch.float16,), (g.rows,)),
            _req(out, "out", (torch.bfloat16,), (g.rows, g.cols)))
    with _on(codes):
        _check("trellis_expand_bf16", load().trellis_expand_bf16(*args, ctypes.byref(g.c()), _stream(codes)))
    return out


def matvec_axis1(codes, scales, x, g: Geometry, out=None, bf16_weights: bool = False):
    """out[M, rows] = x[M, cols] @ W^T for an axis-1 matrix, M = 1..4.

    bf16_weights selects the bf16-rounded weight numerics (the expand weights)."""
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, g.rows), dtype=torch.bfloat16, device=x.device)
    args = (_req(codes, "codes", _CODES, g.codes_shape),
            _req(scales, "scales", (torch.float16,), (g.rows,)),
            _req(x, "x", (torch.bfloat16,), (M, g.cols)),
            _req(out, "out", (torch.bfloat16,), (M, g.rows)))
    fn = "trellis_matvec_axis1_bf16w" if bf16_weights else "trellis_matvec_axis1"
    with _on(x):
        _check(fn, getattr(load(), fn)(*args, M, ctypes.byref(g.c()), _stream(x)))
    return out


def _req_host(t: torch.Tensor, name: str, shape):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} has dtype {t.dtype}, expected torch.bfloat16")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def matvec_axis1_host(codes, scales, x_host, g: Geometry, out_host, x_dev, out_dev):
    """matvec_axis1 with x and out on the host: one C call queues x_host -> x_dev, the matvec and its output's
    transfer to out_host on the current stream of the codes' device.  out_host holds the result once that stream
    has reached the call (synchronize before reading it).  Pinned (16-byte aligned) host tensors are reached
    through their device mapping: a copy kernel fills x_dev and the matvec writes out_host directly, leaving
    out_dev untouched; other host tensors go through copy-engine copies via x_dev and out_dev."""
    M = x_host.shape[0]
    args = (_req(codes, "codes", _CODES, g.codes_shape),
            _req(scales, "scales", (torch.float16,), (g.rows,)),
            _req_host(x_host, "x_host", (M, g.cols)),
            _req_host(out_host, "out_host", (M, g.rows)))
    xd = _req(x_dev, "x_dev", (torch.bfloat16,), (M, g.cols))
    od = _req(out_dev, "out_dev", (torch.bfloat16,), (M, g.rows))
    with _on(codes):
        _check("trellis_matvec_axis1_host",
               load().trellis_matvec_axis1_host(*args, M, ctypes.byref(g.c()), xd, od, _stream(codes)))
    return out_host


def workspace_bytes(M: int, g: Geometry) -> int:
    return int(load().trellis_workspace_bytes(M, ctypes.byref(g.c())))


def new_workspace(M: int, g: Geometry, device) -> torch.Tensor:
    """A zero-filled workspace for matvec_axis0 (reusable across calls)."""
    n = workspace_bytes(M, g)
    if n == 0:
        raise ValueError("unsupported geometry or M for the axis-0 matvec")
    return torch.zeros(((n + 15) // 16) * 4, dtype=torch.int32, device=device)


def matvec_axis0(codes, scales, x, g: Geometry, workspace, out=None, bf16_weights: bool = False):
    """out[M, cols] = x[M, rows] @ W^T for an axis-0 matrix (stored W^T), M = 1..4.

    bf16_weights selects the bf16-rounded weight numerics (the expand weights)."""
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, g.cols), dtype=torch.bfloat16, device=x.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    args = (_req(codes, "codes", _CODES, g.codes_shape),
            _req(scales, "scales", (torch.float16,), (g.rows,)),
            _req(x, "x", (torch.bfloat16,), (M, g.rows)),
            _req(out, "out", (torch.bfloat16,), (M, g.cols)))
    nbytes = workspace.numel() * workspace.element_size()
    fn = "trellis_matvec_axis0_bf16w" if bf16_weights else "trellis_matvec_axis0"
    with _on(x):
        _check(fn, getattr(load(), fn)(*args, M, ctypes.byref(g.c()), workspace.data_ptr(), nbytes, _stream(x)))
    return out


def gateup_swiglu(gcodes, gscales, ucodes, uscales, x, g: Geometry, out=None):
    """out[M, rows] = bf16 SwiGLU chain of the gate and up matvecs, M = 1..4."""
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, g.rows), dtype=torch.bfloat16, device=x.device)
    shp = g.codes_shape
    args = (_req(gcodes, "gcodes", _CODES, shp), _req(gscales, "gscales", (torch.float16,), (g.rows,)),
            _req(ucodes, "ucodes", _CODES, shp), _req(uscales, "uscales", (torch.float16,), (g.rows,)),
            _req(x, "x", (torch.bfloat16,), (M, g.cols)), _req(out, "out", (torch.bfloat16,), (M, g.rows)))
    with _on(x):
        _check("trellis_gateup_swiglu", load().trellis_gateup_swiglu(*args, M, ctypes.byref(g.c()), _stream(x)))
    return out


def gemm_prefill(codes, scales, x, g: Geometry, out=None):
    """Prefill GEMM on the tensor cores with the bf16 expand weights E (stored [rows, cols]):
    axis 1: out[M, rows] = x[M, cols] @ E^T;  axis 0: out[M, cols] = x[M, rows] @ E."""
    M = x.shape[0]
    n_in, n_out = (g.cols, g.rows) if g.axis == 1 else (g.rows, g.cols)
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=x.device)
    args = (_req(codes, "codes", _CODES, g.codes_shape),
            _req(scales, "scales", (torch.float16,), (g.rows,)),
            _req(x, "x", (torch.bfloat16,), (M, n_in)),
            _req(out, "out", (torch.bfloat16,), (M, n_out)))
    with _on(x):
        _check("trellis_gemm_prefill", load().trellis_gemm_prefill(*args, M, ctypes.byref(g.c()), _stream(x)))
    return out


def load_floor(codes: torch.Tensor, g: Geometry, out: torch.Tensor = None, coalesced: bool = False) -> torch.Tensor:
    """Measurement aid: read the axis-1 stream and decode nothing; out[r] = XOR of the words loaded for row r
    (int32 view of uint32).  Default: the M = 1 matvec's access pattern (lane per row); coalesced: a warp per
    row with its lanes on consecutive 16-byte chunks."""
    if out is None:
        out = torch.empty(g.rows, dtype=torch.int32, device=codes.device)
    args = (_req(codes, "codes", _CODES, g.codes_shape), _req(out, "out", (torch.int32,), (g.rows,)))
    fn = "trellis_load_floor_rows" if coalesced else "trellis_load_floor"
    with _on(codes):
        _check(fn, getattr(load(), fn)(*args, ctypes.byref(g.c()), _stream(codes)))
    return out


def prefill_plan(M: int, g: Geometry, sms: int = 0):
    """The tile plan of gemm_prefill (host arithmetic): (tokens per tile, [(first tile, tiles, CTAs per
    tile), ...]).  sms < 1 takes the current device's SM count."""
    bn = ctypes.c_int32(0)
    buf = (ctypes.c_int32 * 6)()
    n = load().trellis_prefill_plan(M, ctypes.byref(g.c()), sms, ctypes.byref(bn), buf)
    _check("trellis_prefill_plan", n if n < 0 else 0)
    return bn.value, [tuple(buf[3 * i:3 * i + 3]) for i in range(n)]


def set_wait_limit(nanoseconds: int = 0) -> None:
    """Diagnostic: limit of each bounded wait of the tensor-core kernel for later launches (0: the default)."""
    _check("trellis_set_wait_limit", load().trellis_set_wait_limit(int(nanoseconds)))


def device_error(reset: bool = False) -> int:
    """Device error word of the tensor-core kernel (0 = no bounded wait gave up)."""
    return int(load().trellis_device_error(1 if reset else 0))


def mlp_decode(gcodes, gscales, ucodes, uscales, dcodes, dscales, x, g_up: Geometry, g_down: Geometry, workspace,
               hidden=None, out=None):
    """Decode-time MLP block: out = down(swiglu(gate(x), up(x))), M = 1..4 (two launches)."""
    M = x.shape[0]
    if hidden is None:
        hidden = torch.empty((M, g_up.rows), dtype=torch.bfloat16, device=x.device)
    if out is None:
        out = torch.empty((M, g_down.cols), dtype=torch.bfloat16, device=x.device)
    shp_u, shp_d = g_up.codes_shape, g_down.codes_shape
    args = (_req(gcodes, "gcodes", _CODES, shp_u), _req(gscales, "gscales", (torch.float16,), (g_up.rows,)),
            _req(ucodes, "ucodes", _CODES, shp_u), _req(uscales, "uscales", (torch.float16,), (g_up.rows,)),
            _req(dcodes, "dcodes", _CODES, shp_d), _req(dscales, "dscales", (torch.float16,), (g_down.rows,)),
            _req(x, "x", (torch.bfloat16,), (M, g_up.cols)), _req(hidden, "hidden", (torch.bfloat16,), (M, g_up.rows)),
            _req(out, "out", (torch.bfloat16,), (M, g_down.cols)))
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    with _on(x):
        _check("trellis_mlp_decode", load().trellis_mlp_decode(*args, M, ctypes.byref(g_up.c()),
                                                              ctypes.byref(g_down.c()), workspace.data_ptr(), nbytes,
                                                              _stream(x)))
    return hidden, out


class MlpDecodeGraph:
    """The decode MLP block captured once into a CUDA graph and replayed.

    Buffers (x, hidden, out, workspace) are fixed at capture time; write the
    next token's activations into `x` and call `replay()`.
    """

    def __init__(self, gcodes, gscales, ucodes, uscales, dcodes, dscales, g_up: Geometry, g_down: Geometry, M: int):
        dev = gcodes.device
        self.x = torch.zeros((M, g_up.cols), dtype=torch.bfloat16, device=dev)
        self.hidden = torch.empty((M, g_up.rows), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((M, g_down.cols), dtype=torch.bfloat16, device=dev)
        self.workspace = new_workspace(M, g_down, dev)
        self._args = (gcodes, gscales, ucodes, uscales, dcodes, dscales)
        self._g = (g_up, g_down)
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):  # warm-up launch outside the graph (library set-up, first-use costs)
            mlp_decode(*self._args, self.x, *self._g, self.workspace, self.hidden, self.out)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            mlp_decode(*self._args, self.x, *self._g, self.workspace, self.hidden, self.out)

    def replay(self):
        self.graph.replay()
        return self.out
