"""CPU oracle for the uniform-grid build — test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
use this package.  It wraps ``grid_oracle.c`` (plain single-threaded C, built
with ``-O2 -ffp-contract=off``, no fast-math) through ctypes and shares no
code with the CUDA library.  Each wrapped function cites its passage in the
C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "grid_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]

_u32p = ctypes.POINTER(ctypes.c_uint32)
_f32p = ctypes.POINTER(ctypes.c_float)


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the oracle C file into a shared library (gcc)."""
    cmd = ["gcc", *CFLAGS, "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def build(force: bool = False) -> str:
    """Build ``liboracle.so`` unless it is newer than its source."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_oracle()
    return LIBRARY


def _ptr(a: np.ndarray, kind):
    return a.ctypes.data_as(kind)


class Oracle:
    """ctypes view of one compiled oracle library (the real one or a test mutant)."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        u64 = ctypes.c_uint64
        u32 = ctypes.c_uint32
        lib.oracle_cell_index.argtypes = [_f32p, u64, _u32p, _f32p, ctypes.c_float, u32, _u32p]
        lib.oracle_histogram.argtypes = [_u32p, u64, _u32p, u64]
        lib.oracle_exclusive_scan.argtypes = [_u32p, u64, _u32p]
        lib.oracle_scatter.argtypes = [_u32p, u64, _u32p, _u32p, u64, _u32p]
        lib.oracle_reorder.argtypes = [_u32p, u64, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_build.argtypes = [_f32p, u64, _u32p, _f32p, ctypes.c_float, u32,
                                     _u32p, _u32p, _u32p, _u32p, _f32p]
        lib.oracle_canonicalise.argtypes = [_u32p, u64, _u32p]
        lib.oracle_diagnostics.argtypes = [_u32p, u64, u64, ctypes.c_uint32, _u32p, _u32p]
        lib.oracle_reorder_records.argtypes = [_u32p, u64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32]
        lib.oracle_density.argtypes = [_f32p, u64, _u32p, _f32p, ctypes.c_float, u32, _u32p, _u32p,
                                       ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_morton_cell.argtypes = [u32, u32, u32, _u32p]
        lib.oracle_morton_cell.restype = u32
        for f in ("oracle_cell_index", "oracle_histogram", "oracle_exclusive_scan",
                  "oracle_scatter", "oracle_reorder", "oracle_build", "oracle_canonicalise",
                  "oracle_diagnostics", "oracle_reorder_records", "oracle_density"):
            getattr(lib, f).restype = None
        self.lib = lib

    # -- one function per step ------------------------------------------------
    def cell_index(self, parts, dims, origin, cell_size, order: int = 0) -> np.ndarray:
        parts = np.ascontiguousarray(parts, dtype=np.float32).reshape(-1, 8)
        dims_a = np.asarray(dims, dtype=np.uint32)
        origin_a = np.asarray(origin, dtype=np.float32)
        out = np.empty(parts.shape[0], dtype=np.uint32)
        self.lib.oracle_cell_index(_ptr(parts, _f32p), parts.shape[0], _ptr(dims_a, _u32p),
                                   _ptr(origin_a, _f32p), float(np.float32(cell_size)), order,
                                   _ptr(out, _u32p))
        return out

    def histogram(self, celda_de, cells: int) -> np.ndarray:
        celda_de = np.ascontiguousarray(celda_de, dtype=np.uint32)
        out = np.empty(cells, dtype=np.uint32)
        self.lib.oracle_histogram(_ptr(celda_de, _u32p), celda_de.size, _ptr(out, _u32p), cells)
        return out

    def exclusive_scan(self, conteos) -> np.ndarray:
        conteos = np.ascontiguousarray(conteos, dtype=np.uint32)
        out = np.empty(conteos.size + 1, dtype=np.uint32)
        self.lib.oracle_exclusive_scan(_ptr(conteos, _u32p), conteos.size, _ptr(out, _u32p))
        return out

    def scatter(self, celda_de, inicios) -> np.ndarray:
        celda_de = np.ascontiguousarray(celda_de, dtype=np.uint32)
        inicios = np.ascontiguousarray(inicios, dtype=np.uint32)
        cells = inicios.size - 1
        cursor = np.empty(cells, dtype=np.uint32)
        out = np.empty(celda_de.size, dtype=np.uint32)
        self.lib.oracle_scatter(_ptr(celda_de, _u32p), celda_de.size, _ptr(inicios, _u32p),
                                _ptr(cursor, _u32p), cells, _ptr(out, _u32p))
        return out

    def reorder(self, ordenado, origen) -> np.ndarray:
        ordenado = np.ascontiguousarray(ordenado, dtype=np.uint32)
        origen = np.ascontiguousarray(origen, dtype=np.float32).reshape(-1, 8)
        out = np.empty((ordenado.size, 8), dtype=np.float32)
        self.lib.oracle_reorder(_ptr(ordenado, _u32p), ordenado.size,
                                origen.ctypes.data_as(ctypes.c_void_p),
                                out.ctypes.data_as(ctypes.c_void_p))
        return out

    def reorder_records(self, ordenado, origen: np.ndarray) -> np.ndarray:
        """destino[k] = origen[ordenado[k]] for one array of equal-size records
        (origen: [N, record_bytes] uint8, or any array whose rows are the records)."""
        ordenado = np.ascontiguousarray(ordenado, dtype=np.uint32)
        src = np.ascontiguousarray(origen)
        rb = src.nbytes // max(src.shape[0], 1) if src.shape[0] else 0
        out = np.empty((ordenado.size,) + src.shape[1:], dtype=src.dtype)
        self.lib.oracle_reorder_records(_ptr(ordenado, _u32p), ordenado.size,
                                        src.ctypes.data_as(ctypes.c_void_p),
                                        out.ctypes.data_as(ctypes.c_void_p), rb)
        return out

    def build(self, parts, dims, origin, cell_size, order: int = 0) -> dict:
        """The whole chain; returns conteos, celdaDe, inicios, ordenado, destino."""
        parts = np.ascontiguousarray(parts, dtype=np.float32).reshape(-1, 8)
        n = parts.shape[0]
        dims_a = np.asarray(dims, dtype=np.uint32)
        origin_a = np.asarray(origin, dtype=np.float32)
        cells = int(dims_a[0]) * int(dims_a[1]) * int(dims_a[2])
        out = {
            "conteos": np.empty(cells, dtype=np.uint32),
            "celdaDe": np.empty(n, dtype=np.uint32),
            "inicios": np.empty(cells + 1, dtype=np.uint32),
            "ordenado": np.empty(n, dtype=np.uint32),
            "destino": np.empty((n, 8), dtype=np.float32),
        }
        self.lib.oracle_build(_ptr(parts, _f32p), n, _ptr(dims_a, _u32p), _ptr(origin_a, _f32p),
                              float(np.float32(cell_size)), order, _ptr(out["conteos"], _u32p),
                              _ptr(out["celdaDe"], _u32p), _ptr(out["inicios"], _u32p),
                              _ptr(out["ordenado"], _u32p), _ptr(out["destino"], _f32p))
        return out

    def diagnostics(self, celda_de, cells: int, capacidad: int = 64) -> tuple[int, int]:
        """(maxPorCelda, desbordes) while counting the particles in index order."""
        celda_de = np.ascontiguousarray(celda_de, dtype=np.uint32)
        cursor = np.empty(max(cells, 1), dtype=np.uint32)
        diag = np.zeros(2, dtype=np.uint32)
        self.lib.oracle_diagnostics(_ptr(celda_de, _u32p), celda_de.size, cells, capacidad,
                                    _ptr(cursor, _u32p), _ptr(diag, _u32p))
        return int(diag[0]), int(diag[1])

    def density(self, parts, dims, origin, cell_size, inicios, ordenado, h: float, order: int = 0) -> np.ndarray:
        """rho[i] (float64) for every particle i of `parts` (original order),
        walking the 27 cells around it through inicios / ordenado."""
        parts = np.ascontiguousarray(parts, dtype=np.float32).reshape(-1, 8)
        dims_a = np.asarray(dims, dtype=np.uint32)
        origin_a = np.asarray(origin, dtype=np.float32)
        inicios = np.ascontiguousarray(inicios, dtype=np.uint32)
        ordenado = np.ascontiguousarray(ordenado, dtype=np.uint32)
        out = np.empty(parts.shape[0], dtype=np.float64)
        self.lib.oracle_density(_ptr(parts, _f32p), parts.shape[0], _ptr(dims_a, _u32p), _ptr(origin_a, _f32p),
                                float(np.float32(cell_size)), order, _ptr(inicios, _u32p), _ptr(ordenado, _u32p),
                                float(h), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
        return out

    def morton_cell(self, x: int, y: int, z: int, dims) -> int:
        dims_a = np.asarray(dims, dtype=np.uint32)
        return int(self.lib.oracle_morton_cell(x, y, z, _ptr(dims_a, _u32p)))

    def canonicalise(self, inicios, ordenado) -> np.ndarray:
        """Copy of ordenado with every cell segment sorted ascending."""
        inicios = np.ascontiguousarray(inicios, dtype=np.uint32)
        out = np.array(ordenado, dtype=np.uint32, copy=True)
        self.lib.oracle_canonicalise(_ptr(inicios, _u32p), inicios.size - 1, _ptr(out, _u32p))
        return out


_DEFAULT: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``grid_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(build())
    return _DEFAULT
