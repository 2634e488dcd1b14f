"""Python binding of libugrid: the C ABI's entry points under the same names.

Argument marshalling only: each function checks the tensors' device, dtype,
shape and contiguity, passes their device pointers and the current CUDA
stream to the C ABI, and raises ``GridError`` on a non-zero status.  Every
step of the build runs in the library's CUDA kernels; there is no fallback.
PyTorch provides the device memory and the streams.

Tensor conventions: particle arrays are float32 ``[N, 8]`` (the 32-byte
Particula rows); u32 arrays are int32 or uint32 tensors of the stated length
(reinterpreted as u32).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np
import torch

from . import build as _build

GRID_OK, GRID_EINVAL, GRID_ECUDA, GRID_ETIMEOUT, GRID_EBOUNDS, GRID_ERANGE = 0, 1, 2, 3, 4, 5
GRID_STABLE = 1

_U32_DTYPES = (torch.int32, getattr(torch, "uint32", torch.int32))


class GridError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (status {code})")


class grid_params(ctypes.Structure):
    """Mirror of ``grid_params`` in include/ugrid.h."""

    _fields_ = [
        ("conteo", ctypes.c_uint32),
        ("celdas", ctypes.c_uint32),
        ("dims", ctypes.c_uint32 * 3),
        ("origin", ctypes.c_float * 3),
        ("cellSize", ctypes.c_float),
        ("order", ctypes.c_uint32),
    ]


GRID_ORDER_LINEAR = 0
GRID_ORDER_MORTON = 1


class grid_array(ctypes.Structure):
    """Mirror of ``grid_array`` in include/ugrid.h."""

    _fields_ = [("origen", ctypes.c_void_p), ("destino", ctypes.c_void_p), ("record_bytes", ctypes.c_uint32)]


def make_params(n: int, dims, origin, cell_size: float, order: int = GRID_ORDER_LINEAR) -> grid_params:
    p = grid_params()
    p.order = int(order)
    p.conteo = int(n)
    p.dims[:] = [int(d) for d in dims]
    p.celdas = int(dims[0]) * int(dims[1]) * int(dims[2]) & 0xFFFFFFFF
    p.origin[:] = [float(np.float32(o)) for o in origin]
    p.cellSize = float(np.float32(cell_size))
    return p


_lib = None


def library_path() -> str:
    return _build.LIBRARY


def lib() -> ctypes.CDLL:
    """The loaded libugrid.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m uniform_grid_particle_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(path)
        vp, pp, u = ctypes.c_void_p, ctypes.POINTER(grid_params), ctypes.c_uint
        sigs = {
            "grid_workspace_bytes": ([pp, u], ctypes.c_size_t),
            "grid_workspace_init": ([vp, ctypes.c_size_t, vp], ctypes.c_int),
            "grid_clear": ([vp, pp, vp], ctypes.c_int),
            "grid_count": ([vp, vp, vp, pp, vp], ctypes.c_int),
            "grid_scan": ([vp, vp, vp, pp, vp], ctypes.c_int),
            "grid_scatter": ([vp, vp, vp, vp, u, vp, pp, vp], ctypes.c_int),
            "grid_reorder": ([vp, vp, vp, vp, pp, vp], ctypes.c_int),
            "grid_build": ([vp, vp, vp, vp, vp, vp, vp, u, pp, vp], ctypes.c_int),
            "grid_build_host": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u, pp, vp], ctypes.c_int),
            "grid_status": ([vp, vp], ctypes.c_int),
            "grid_scan_noalloc": ([vp, vp, pp, vp], ctypes.c_int),
            "grid_diagnostics": ([vp, ctypes.c_uint32, vp, pp, vp], ctypes.c_int),
            "grid_density": ([vp, vp, vp, ctypes.c_float, vp, vp, pp, vp], ctypes.c_int),
            "grid_reorder_many": ([vp, ctypes.POINTER(grid_array), ctypes.c_uint32, vp, pp, vp], ctypes.c_int),
            "grid_error_string": ([ctypes.c_int], ctypes.c_char_p),
        }
        for name, (args, res) in sigs.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def error_string(code: int) -> str:
    return lib().grid_error_string(code).decode()


def _check(code: int, where: str) -> None:
    if code != GRID_OK:
        raise GridError(code, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, name: str, numel: int, dtypes) -> int | None:
    if t is None:
        if numel == 0:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr() or None


def _u32(t, name, numel):
    return _ptr(t, name, numel, _U32_DTYPES)


def _parts(t, name, n):
    if t is not None and t.dim() == 2 and t.shape[1] != 8:
        raise ValueError(f"{name} must be float32 [N, 8]")
    return _ptr(t, name, 8 * n, (torch.float32,))


def _ws(t, name="ws"):
    return _ptr(t, name, 1, (torch.uint8,))


# ---- entry points (same names as the C ABI) --------------------------------

def grid_workspace_bytes(p: grid_params, flags: int = 0) -> int:
    return int(lib().grid_workspace_bytes(ctypes.byref(p), flags))


def grid_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib().grid_workspace_init(_ws(ws), ws.numel(), _stream(stream)), "grid_workspace_init")


def grid_clear(conteos, p: grid_params, stream=None) -> None:
    _check(lib().grid_clear(_u32(conteos, "conteos", p.celdas), ctypes.byref(p), _stream(stream)),
           "grid_clear")


def grid_count(parts, conteos, celdaDe, p: grid_params, stream=None) -> None:
    _check(lib().grid_count(_parts(parts, "parts", p.conteo), _u32(conteos, "conteos", p.celdas),
                            _u32(celdaDe, "celdaDe", p.conteo), ctypes.byref(p), _stream(stream)),
           "grid_count")


def grid_scan(conteos, inicios, ws, p: grid_params, stream=None) -> None:
    _check(lib().grid_scan(_u32(conteos, "conteos", p.celdas), _u32(inicios, "inicios", p.celdas + 1),
                           _ws(ws), ctypes.byref(p), _stream(stream)), "grid_scan")


def grid_scatter(celdaDe, inicios, cursor, ordenado, ws, p: grid_params, flags: int = 0,
                 stream=None) -> None:
    _check(lib().grid_scatter(_u32(celdaDe, "celdaDe", p.conteo), _u32(inicios, "inicios", p.celdas + 1),
                              _u32(cursor, "cursor", p.celdas), _u32(ordenado, "ordenado", p.conteo),
                              flags, _ws(ws), ctypes.byref(p), _stream(stream)), "grid_scatter")


def grid_reorder(ordenado, origen, destino, ws, p: grid_params, stream=None) -> None:
    _check(lib().grid_reorder(_u32(ordenado, "ordenado", p.conteo), _parts(origen, "origen", p.conteo),
                              _parts(destino, "destino", p.conteo), _ws(ws), ctypes.byref(p),
                              _stream(stream)), "grid_reorder")


def grid_build(origen, destino, conteos, celdaDe, inicios, ordenado, ws, p: grid_params,
               flags: int = 0, stream=None) -> None:
    _check(lib().grid_build(_parts(origen, "origen", p.conteo), _parts(destino, "destino", p.conteo),
                            _u32(conteos, "conteos", p.celdas), _u32(celdaDe, "celdaDe", p.conteo),
                            _u32(inicios, "inicios", p.celdas + 1), _u32(ordenado, "ordenado", p.conteo),
                            _ws(ws), flags, ctypes.byref(p), _stream(stream)), "grid_build")


def _host(t, name, numel, dtypes):
    """A CPU tensor's data pointer (page-locked memory keeps the copies asynchronous)."""
    if t is None:
        if numel == 0:
            return None
        raise ValueError(f"{name} is required")
    if t.is_cuda or t.dtype not in dtypes or not t.is_contiguous() or t.numel() < numel:
        raise ValueError(f"{name} must be a contiguous CPU tensor of {dtypes} with at least {numel} elements")
    return t.data_ptr()


def grid_build_host(origen_host, destino_host, inicios_host, origen, destino, conteos, celdaDe, inicios, ordenado,
                    ws, p: grid_params, flags: int = 0, stream=None) -> None:
    """grid_build between host arrays: origen_host is copied to origen, the
    grid is built, destino and inicios are copied back, all on the stream."""
    n, c = int(p.conteo), int(p.celdas)
    _check(lib().grid_build_host(_host(origen_host, "origen_host", 8 * n, (torch.float32,)),
                                 _host(destino_host, "destino_host", 8 * n, (torch.float32,)),
                                 _host(inicios_host, "inicios_host", c + 1, _U32_DTYPES),
                                 _parts(origen, "origen", n), _parts(destino, "destino", n),
                                 _u32(conteos, "conteos", c), _u32(celdaDe, "celdaDe", n),
                                 _u32(inicios, "inicios", c + 1), _u32(ordenado, "ordenado", n),
                                 _ws(ws), flags, ctypes.byref(p), _stream(stream)), "grid_build_host")


def grid_scan_noalloc(conteos, inicios, p: grid_params, stream=None) -> None:
    """The scan of grid_scan for callers that cannot allocate: its scratch is a
    fixed array inside the library (at most 33,554,432 cells; calls that
    overlap on the GPU race on it)."""
    _check(lib().grid_scan_noalloc(_u32(conteos, "conteos", p.celdas),
                                   _u32(inicios, "inicios", p.celdas + 1), ctypes.byref(p),
                                   _stream(stream)), "grid_scan_noalloc")


def grid_reorder_many(ordenado, pairs, ws, p: grid_params, stream=None) -> None:
    """pairs: list of (origen, destino) CUDA tensors with N rows each; every
    row of an array is one record (its byte size a multiple of 16)."""
    if not 1 <= len(pairs) <= 4:
        raise ValueError("between 1 and 4 arrays")
    descs = (grid_array * len(pairs))()
    n = int(p.conteo)
    for d, (src, dst) in zip(descs, pairs):
        for t, name in ((src, "origen"), (dst, "destino")):
            if not t.is_cuda or not t.is_contiguous() or t.shape[0] != n:
                raise ValueError(f"{name} must be a contiguous CUDA tensor with {n} rows")
        if src.dtype != dst.dtype or src.shape != dst.shape:
            raise ValueError("origen and destino must have the same dtype and shape")
        d.origen = src.data_ptr() or None
        d.destino = dst.data_ptr() or None
        d.record_bytes = (src.numel() * src.element_size()) // n if n else 16
    _check(lib().grid_reorder_many(_u32(ordenado, "ordenado", n), descs, len(pairs), _ws(ws), ctypes.byref(p),
                                   _stream(stream)), "grid_reorder_many")


def grid_density(parts, inicios, rho, ws, p: grid_params, h: float, ordenado=None, stream=None) -> None:
    """rho[k] for the particle at cell-order position k: parts is destino when
    ordenado is None, else origen read through ordenado."""
    _check(lib().grid_density(_parts(parts, "parts", p.conteo),
                              None if ordenado is None else _u32(ordenado, "ordenado", p.conteo),
                              _u32(inicios, "inicios", p.celdas + 1), float(np.float32(h)),
                              _ptr(rho, "rho", p.conteo, (torch.float32,)), _ws(ws), ctypes.byref(p),
                              _stream(stream)), "grid_density")


def grid_diagnostics(conteos, diag, p: grid_params, capacidad: int = 64, stream=None) -> None:
    """diag[0] = maxPorCelda, diag[1] = desbordes for the given capacity."""
    _check(lib().grid_diagnostics(_u32(conteos, "conteos", p.celdas), capacidad, _u32(diag, "diag", 2),
                                  ctypes.byref(p), _stream(stream)), "grid_diagnostics")


def grid_status(ws, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().grid_status(_ws(ws), _stream(stream)))


# ---- convenience: caller-owned buffers for one grid -------------------------

@dataclasses.dataclass
class GridBuffers:
    """Device arrays of one grid build, allocated by PyTorch (the caller)."""

    conteos: torch.Tensor
    celdaDe: torch.Tensor
    inicios: torch.Tensor
    ordenado: torch.Tensor
    destino: torch.Tensor
    ws: torch.Tensor

    @classmethod
    def allocate(cls, p: grid_params, flags: int = 0, device="cuda") -> "GridBuffers":
        n, c = int(p.conteo), int(p.celdas)
        ws_bytes = grid_workspace_bytes(p, flags)
        if ws_bytes == 0:
            raise GridError(GRID_EINVAL, "grid_workspace_bytes")
        i32 = dict(dtype=torch.int32, device=device)
        return cls(
            conteos=torch.empty(c, **i32),
            celdaDe=torch.empty(n, **i32),
            inicios=torch.empty(c + 1, **i32),
            ordenado=torch.empty(n, **i32),
            destino=torch.empty((n, 8), dtype=torch.float32, device=device),
            ws=torch.zeros(ws_bytes, dtype=torch.uint8, device=device),
        )

    def build(self, origen: torch.Tensor, p: grid_params, flags: int = 0, stream=None) -> None:
        grid_build(origen, self.destino, self.conteos, self.celdaDe, self.inicios, self.ordenado,
                   self.ws, p, flags, stream)
