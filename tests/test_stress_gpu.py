"""Stress workload: 16,777,216 particles on 256^3 cells, ten builds in a row
with origen and destino swapped after each ("El estado de las partículas en
storage buffers", §Doble buffer: two buffers that alternate).

The positions do not change between builds, so after the first build the
records are already grouped by cell: every later build must find the
identity order (after canonicalisation; exactly in stable mode) and copy the
records unchanged.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import to_u32
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    return ugrid


@pytest.mark.parametrize("stable", [False, True], ids=["atomic", "stable"])
def test_ten_ping_pong_builds(ug, oracle_lib, stable):
    s = scenes.SCENES["stress"]
    rows = s.particles()
    flags = ug.GRID_STABLE if stable else 0
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
    b = ug.GridBuffers.allocate(p, flags)
    bufs = [torch.from_numpy(rows).cuda(), b.destino]
    ref = oracle_lib.build(rows, s.dims, s.origin, s.cell_size)
    identity = np.arange(s.n, dtype=np.uint32)
    for k in range(s.builds):
        origen, destino = bufs[k % 2], bufs[(k + 1) % 2]
        ug.grid_build(origen, destino, b.conteos, b.celdaDe, b.inicios, b.ordenado, b.ws, p, flags)
        assert ug.grid_status(b.ws) == 0
        inicios = to_u32(b.inicios)
        ordenado = to_u32(b.ordenado)
        assert np.array_equal(inicios, ref["inicios"]), f"build {k + 1}: inicios"
        assert np.array_equal(to_u32(b.conteos), ref["conteos"]), f"build {k + 1}: conteos"
        if k == 0:
            assert np.array_equal(to_u32(b.celdaDe), ref["celdaDe"])
            want = ref["ordenado"]
            got = ordenado if stable else oracle_lib.canonicalise(inicios, ordenado)
            assert np.array_equal(got, want)
            dest = destino.cpu().numpy()
            assert np.array_equal(dest.view(np.uint32), rows.view(np.uint32)[ordenado])
            if stable:
                assert np.array_equal(dest.view(np.uint32), ref["destino"].view(np.uint32))
        else:
            celda = to_u32(b.celdaDe)
            assert np.all(np.diff(celda.astype(np.int64)) >= 0), f"build {k + 1}: celdaDe not sorted"
            got = ordenado if stable else oracle_lib.canonicalise(inicios, ordenado)
            assert np.array_equal(got, identity), f"build {k + 1}: order is not the identity"
            if stable or k == s.builds - 1:
                src = origen.cpu().numpy().view(np.uint32)
                dst = destino.cpu().numpy().view(np.uint32)
                if stable:
                    assert np.array_equal(dst, src), f"build {k + 1}: records changed"
                else:
                    assert np.array_equal(dst, src[ordenado])
    final = bufs[s.builds % 2].cpu().numpy()
    assert np.array_equal(np.sort(final.view(np.uint32), axis=0), np.sort(rows.view(np.uint32), axis=0))
