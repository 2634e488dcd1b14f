"""Rows beyond the core build: overflow diagnostics and the multi-array gather,
through the C ABI, against the CPU oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu_build, to_u32
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    return ugrid


@pytest.mark.parametrize("name", ["headline", "contention", "tiny"])
@pytest.mark.parametrize("capacidad", [1, 4, 64, 100_000])
def test_diagnostics_match_oracle(ug, oracle_lib, name, capacidad):
    s = scenes.SCENES[name]
    rows = s.particles()
    got = gpu_build(ug, rows, s.dims, s.origin, s.cell_size)
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
    diag = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    ug.grid_diagnostics(torch.from_numpy(got["conteos"].view(np.int32)).cuda(), diag, p, capacidad)
    want = oracle_lib.diagnostics(oracle_lib.cell_index(rows, s.dims, s.origin, s.cell_size), s.cells, capacidad)
    assert tuple(int(v) for v in to_u32(diag)) == want


def test_diagnostics_ragged_cells(ug, oracle_lib):
    dims = (7, 11, 13)                       # 1001 cells: not a multiple of 4
    rng = np.random.default_rng(3)
    celda = rng.integers(0, 1001, 50_000, dtype=np.uint32)
    celda[:3000] = 1000                      # the last cell, in the tail of the vector loop
    conteos = np.bincount(celda, minlength=1001).astype(np.uint32)
    p = ug.make_params(celda.size, dims, (0, 0, 0), 1.0)
    diag = torch.empty(2, dtype=torch.int32, device="cuda")
    ug.grid_diagnostics(torch.from_numpy(conteos.view(np.int32)).cuda(), diag, p, 64)
    assert tuple(int(v) for v in to_u32(diag)) == oracle_lib.diagnostics(celda, 1001, 64)


def test_reorder_many_matches_oracle(ug, oracle_lib):
    s = scenes.SCENES["headline"]
    rows = s.particles()
    got = gpu_build(ug, rows, s.dims, s.origin, s.cell_size)
    ordenado = got["ordenado"]
    n = s.n
    rng = np.random.default_rng(9)
    aspecto = rng.integers(0, 2**32, (n, 8), dtype=np.uint64).astype(np.uint32)     # color, tam, semilla, _r
    wide = rng.integers(0, 2**32, (n, 12), dtype=np.uint64).astype(np.uint32)       # 48-byte records
    narrow = rng.integers(0, 2**32, (n, 4), dtype=np.uint64).astype(np.uint32)      # 16-byte records
    hosts = [rows, aspecto, wide, narrow]
    srcs = [torch.from_numpy(h).cuda() for h in hosts]
    dsts = [torch.empty_like(t) for t in srcs]
    p = ug.make_params(n, s.dims, s.origin, s.cell_size)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ug.grid_reorder_many(torch.from_numpy(ordenado.view(np.int32)).cuda(), list(zip(srcs, dsts)), ws, p)
    assert ug.grid_status(ws) == 0
    for h, d in zip(hosts, dsts):
        want = oracle_lib.reorder_records(ordenado, h)
        assert np.array_equal(d.cpu().numpy().view(np.uint8), want.view(np.uint8))
    # the particle array matches the build's own gather
    assert np.array_equal(dsts[0].cpu().numpy().view(np.uint32), got["destino"].view(np.uint32))


def test_reorder_many_rejects_index_out_of_range(ug):
    n = 2000
    p = ug.make_params(n, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    ordenado = torch.randperm(n, device="cuda").int()
    ordenado[5] = n
    a, b = torch.randn(n, 8, device="cuda"), torch.randn(n, 4, device="cuda")
    da, db = torch.zeros_like(a), torch.zeros_like(b)
    ug.grid_reorder_many(ordenado, [(a, da), (b, db)], ws, p)
    assert ug.grid_status(ws) == 4
    assert (da[5] == 0).all() and (db[5] == 0).all()
    ok = torch.arange(n, device="cuda") != 5
    assert torch.equal(da[ok], a[ordenado[ok].long()]) and torch.equal(db[ok], b[ordenado[ok].long()])
