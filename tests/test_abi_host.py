"""The C-ABI library without a GPU: it loads, exports every declared symbol,
sizes its workspace, and rejects bad arguments before any CUDA call."""
import ctypes
import math
import os
import re
import subprocess

import pytest

from uniform_grid_particle_gb300 import build as ugbuild

HEADER = os.path.join(ugbuild.INCLUDE, "ugrid.h")
EINVAL = 1


@pytest.fixture(scope="module")
def L():
    ugbuild.build()
    from uniform_grid_particle_gb300 import ugrid

    return ugrid


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(grid_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10, names
    lib = ctypes.CDLL(L.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def P(L, n=1000, dims=(16, 16, 16), origin=(-5, -5, -5), cs=0.625):
    return L.make_params(n, dims, origin, cs)


def test_workspace_bytes(L):
    p = P(L, 1_000_000, (128, 128, 128), cs=0.078125)
    tiles = (128 ** 3 + 8191) // 8192       # scan tiles of 8192 cells
    r256 = lambda b: (b + 255) // 256 * 256                     # noqa: E731
    # The arrays that stay zero between calls, at offsets that do not depend on
    # the particle count: header (alone in 4 KB), bucket totals (8192 buckets x 8 lane words),
    # look-back words, per-cell counters.  Then scratch: per-CTA chunk sums (up
    # to 4096 CTAs), bucket bases, per-particle slots and (cell, particle) pairs.
    fixed = 4096 + r256(4 * 8 * 8192)   # the header padded to 4 KB
    assert L.grid_workspace_bytes(p, 0) == (fixed + r256(tiles * 8 * 16) + r256(4 * 128 ** 3) + r256(4096 * 4)
                                            + r256(4 * 8192) + r256(4 * 1_000_000) + r256(8 * 1_000_000))
    stable = L.grid_workspace_bytes(p, L.GRID_STABLE)
    assert stable >= L.grid_workspace_bytes(p, 0) + 4 * 1_000_000
    assert L.grid_workspace_bytes(p, 2) == 0            # unknown flag
    bad = P(L)
    bad.celdas = 7
    assert L.grid_workspace_bytes(bad, 0) == 0
    tiny = P(L, 0, (1, 1, 1), cs=1.0)
    assert L.grid_workspace_bytes(tiny, 0) == fixed + 256 + 256 + 4096 * 4 + 4 * 8192


def test_error_strings(L):
    for code in range(6):
        assert L.error_string(code)


FAKE = 0x7F0000000000          # 256-aligned, never dereferenced: every call below fails validation


def _call(L, name, *args):
    return getattr(L.lib(), name)(*args)


@pytest.mark.parametrize("mutate", [
    lambda p: setattr(p, "celdas", p.celdas + 1),
    lambda p: p.dims.__setitem__(0, 0),
    lambda p: setattr(p, "cellSize", 0.0),
    lambda p: setattr(p, "cellSize", -1.0),
    lambda p: setattr(p, "cellSize", math.nan),
    lambda p: setattr(p, "cellSize", math.inf),
    lambda p: setattr(p, "cellSize", 1e-45),          # 1/cellSize overflows to inf
    lambda p: p.origin.__setitem__(1, math.nan),
    lambda p: p.origin.__setitem__(2, -math.inf),
    lambda p: setattr(p, "order", 2),
    lambda p: (setattr(p, "order", 1), p.dims.__setitem__(1, 3), setattr(p, "celdas", p.dims[0] * 3 * p.dims[2])),
], ids=["celdas", "dims0", "cs0", "cs_neg", "cs_nan", "cs_inf", "cs_denorm", "origin_nan", "origin_inf",
        "order_unknown", "morton_not_pow2"])
def test_bad_params_rejected_everywhere(L, mutate):
    p = P(L)
    mutate(p)
    bp = ctypes.byref(p)
    f = FAKE
    assert _call(L, "grid_clear", f, bp, None) == EINVAL
    assert _call(L, "grid_count", f, f + (1 << 30), f + (2 << 30), bp, None) == EINVAL
    assert _call(L, "grid_scan", f, f + (1 << 30), f + (2 << 30), bp, None) == EINVAL
    assert _call(L, "grid_scatter", f, f + (1 << 30), f + (2 << 30), f + (3 << 30), 0, f + (4 << 30), bp, None) == EINVAL
    assert _call(L, "grid_reorder", f, f + (1 << 30), f + (2 << 30), f + (3 << 30), bp, None) == EINVAL
    assert _call(L, "grid_build", f, f + (1 << 30), f + (2 << 30), f + (3 << 30), f + (4 << 30),
                 f + (5 << 30), f + (6 << 30), 0, bp, None) == EINVAL


def test_cell_count_overflow_rejected(L):
    p = P(L, 10, (65536, 65536, 1), cs=1.0)     # 2^32 cells: C + 1 would not fit in u32
    assert L.grid_workspace_bytes(p, 0) == 0
    p = P(L, 10, (65535, 65537, 1), cs=1.0)     # 2^32 - 1 cells: the largest rejected
    assert L.grid_workspace_bytes(p, 0) == 0
    p = P(L, 10, (2, 3, 4), cs=1.0)
    p.dims[:] = [4294967295, 4294967295, 4294967295]
    p.celdas = 1
    assert L.grid_workspace_bytes(p, 0) == 0


def test_null_params_and_pointers(L):
    f = FAKE
    assert _call(L, "grid_clear", f, None, None) == EINVAL
    assert L.lib().grid_workspace_bytes(None, 0) == 0
    p = P(L)
    bp = ctypes.byref(p)
    assert _call(L, "grid_clear", None, bp, None) == EINVAL
    assert _call(L, "grid_count", None, f, f + (1 << 30), bp, None) == EINVAL
    assert _call(L, "grid_reorder", f, f + (1 << 30), f + (2 << 30), None, bp, None) == EINVAL
    assert _call(L, "grid_status", None, None) == EINVAL
    assert _call(L, "grid_workspace_init", None, 4096, None) == EINVAL


def test_alignment_rules(L):
    p = P(L)
    bp = ctypes.byref(p)
    f = FAKE
    # particles must be 16-byte aligned, conteos 16, celdaDe 4
    assert _call(L, "grid_count", f + 8, f + (1 << 30), f + (2 << 30), bp, None) == EINVAL
    assert _call(L, "grid_count", f, f + (1 << 30) + 4, f + (2 << 30), bp, None) == EINVAL
    assert _call(L, "grid_count", f, f + (1 << 30), f + (2 << 30) + 2, bp, None) == EINVAL
    # the workspace must be 256-byte aligned
    assert _call(L, "grid_scan", f, f + (1 << 30), f + (2 << 30) + 16, bp, None) == EINVAL
    assert _call(L, "grid_workspace_init", f + 16, 4096, None) == EINVAL


def test_overlapping_buffers_rejected(L):
    p = P(L, 1000)
    bp = ctypes.byref(p)
    f = FAKE
    # destino overlapping origen (in-place gather is refused)
    assert _call(L, "grid_reorder", f + (3 << 30), f, f + 1024, f + (4 << 30), bp, None) == EINVAL
    assert _call(L, "grid_reorder", f + (3 << 30), f, f, f + (4 << 30), bp, None) == EINVAL
    # inicios overlapping conteos in the scan
    assert _call(L, "grid_scan", f, f + 4096, f + (2 << 30), bp, None) == EINVAL
    # cursor aliasing celdaDe in the scatter
    assert _call(L, "grid_scatter", f, f + (1 << 30), f, f + (3 << 30), 0, f + (4 << 30), bp, None) == EINVAL
    # unknown flag bits
    assert _call(L, "grid_scatter", f, f + (1 << 30), f + (2 << 30), f + (3 << 30), 4, f + (4 << 30), bp, None) == EINVAL


def test_binding_checks_tensors_before_the_library(L):
    import torch

    p = P(L, 10)
    with pytest.raises(ValueError):
        L.grid_clear(torch.zeros(4096, dtype=torch.int32), p)          # CPU tensor


def test_reorder_many_and_diagnostics_validation(L):
    p = P(L, 1000)
    bp = ctypes.byref(p)
    f = FAKE
    lib = L.lib()
    A = L.grid_array

    def many(*specs, count=None):
        arr = (A * max(len(specs), 1))()
        for d, (src, dst, rb) in zip(arr, specs):
            d.origen, d.destino, d.record_bytes = src, dst, rb
        return lib.grid_reorder_many(f, arr, len(specs) if count is None else count, f + (1 << 34), bp, None)

    assert many((f + (1 << 30), f + (2 << 30), 32), count=0) == EINVAL          # no arrays
    assert many(*[(f + (i << 30), f + ((i + 8) << 30), 32) for i in range(1, 6)]) == EINVAL   # five arrays
    assert many((f + (1 << 30), f + (2 << 30), 24)) == EINVAL                   # not a multiple of 16
    assert many((f + (1 << 30), f + (2 << 30), 512)) == EINVAL                  # above 256 bytes
    assert many((f + (1 << 30) + 8, f + (2 << 30), 32)) == EINVAL               # misaligned origen
    assert many((f + (1 << 30), f + (1 << 30) + 64, 32)) == EINVAL              # destino inside its origen
    assert many((f + (1 << 30), f + (2 << 30), 32), (f + (3 << 30), f + (2 << 30), 32)) == EINVAL  # shared destino
    assert many((f + (1 << 30), f + (2 << 30), 32), (f + (2 << 30), f + (3 << 30), 32)) == EINVAL  # destino is another origen
    assert lib.grid_diagnostics(f, 64, None, bp, None) == EINVAL
    assert lib.grid_diagnostics(f, 64, f, bp, None) == EINVAL                   # diag inside conteos


def test_density_radius_rules(L):
    p = P(L, 1000, cs=0.625)
    bp = ctypes.byref(p)
    f = FAKE
    lib = L.lib()
    for h in (0.0, -0.1, 0.7, math.nan, math.inf):       # must be 0 < h <= cellSize
        assert lib.grid_density(f, None, f + (1 << 30), h, f + (2 << 30), f + (3 << 30), bp, None) == EINVAL
    assert lib.grid_density(f, f, f + (1 << 30), 0.5, f + (2 << 30), f + (3 << 30), bp, None) == EINVAL  # ordenado inside parts


def test_morton_accepts_power_of_two_sides(L):
    """Morton order takes any power-of-two sides, unequal and of size 1 included."""
    for dims in ((4, 4, 4), (8, 2, 16), (1, 1, 1), (1024, 1024, 1024), (2, 1, 1 << 20)):
        p = L.make_params(10, dims, (0.0, 0.0, 0.0), 1.0, order=L.GRID_ORDER_MORTON)
        assert L.grid_workspace_bytes(p, 0) > 0, dims
    p = L.make_params(10, (4, 4, 6), (0.0, 0.0, 0.0), 1.0, order=L.GRID_ORDER_MORTON)
    assert L.grid_workspace_bytes(p, 0) == 0


def test_build_host_checks_host_arrays(L):
    """grid_build_host rejects missing or overlapping host arrays, and bad
    device arrays, before anything is enqueued."""
    p = P(L)
    bp = ctypes.byref(p)
    f = FAKE
    dev = [f + (k << 30) for k in range(3, 10)]      # origen .. ws, all distinct and aligned
    h = 0x100000000                                  # host addresses, never dereferenced
    call = lambda oh, dh, ih, d=dev: _call(L, "grid_build_host", oh, dh, ih, *d, 0, bp, None)  # noqa: E731
    assert call(None, h + (1 << 24), h + (2 << 24)) == EINVAL          # no origen_host
    assert call(h, None, h + (2 << 24)) == EINVAL                      # no destino_host
    assert call(h, h + (1 << 24), None) == EINVAL                      # no inicios_host
    assert call(h, h + 64, h + (2 << 24)) == EINVAL                    # destino_host inside origen_host
    assert call(h, h + (1 << 24), h + (1 << 24) + 32) == EINVAL        # inicios_host inside destino_host
    bad = list(dev)
    bad[0] = dev[0] + 8                                                 # misaligned device origen
    assert call(h, h + (1 << 24), h + (2 << 24), bad) == EINVAL


def test_workspace_header_layout(tmp_path):
    """The header words that the GPU fault tests write by index sit where the
    tests expect them, as the C compiler lays the struct out: the status word
    first, bar_exit at word 5, bar_extra at word 8, the barrier counter alone
    at word 32, 256 bytes in all."""
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include "ugrid.h"\n'
                   "int main(void) {\n"
                   '  printf("%zu %zu %zu %zu %zu %zu\\n", offsetof(grid_ws_header, status),\n'
                   "         offsetof(grid_ws_header, scan_ticket), offsetof(grid_ws_header, bar_exit),\n"
                   "         offsetof(grid_ws_header, bar_extra), offsetof(grid_ws_header, bar_count),\n"
                   "         sizeof(grid_ws_header));\n"
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", ugbuild.INCLUDE, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert [int(v) for v in out] == [0, 4, 5 * 4, 8 * 4, 32 * 4, 256]
