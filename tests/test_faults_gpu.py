"""Device-detected problems come back as status codes and leave the GPU usable.

No test here faults, traps or hangs the GPU: the waits that run out are the
scan's look-back on a tile that no CTA was given and the single-launch
builds' grid barriers with their target raised past the CTA count (each
wait's one-second limit ends it), and the out-of-range indices are caught by
the kernels' own bounds checks before any access.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import to_u32
from uniform_grid_particle_gb300 import scenes

pytestmark = pytest.mark.gpu

ETIMEOUT, EBOUNDS = 3, 4


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    return ugrid


def test_lookback_wait_times_out_and_workspace_recovers(ug, oracle_lib):
    dims = (64, 64, 16)                      # 65536 cells = 8 scan tiles
    C = 64 * 64 * 16
    rng = np.random.default_rng(1)
    conteos = rng.integers(0, 5, C, dtype=np.uint32)
    p = ug.make_params(int(conteos.sum()), dims, (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    inicios = torch.empty(C + 1, dtype=torch.int32, device="cuda")
    dev_conteos = torch.from_numpy(conteos.view(np.int32)).cuda()
    # Start the tile tickets at 1: tile 0 is never taken, so its look-back word
    # is never published and the waits on it run out.
    ws.view(torch.int32)[1] = 1
    ug.grid_scan(dev_conteos, inicios, ws, p)
    assert ug.grid_status(ws) == ETIMEOUT
    header = ws[:256].view(torch.int32).cpu().numpy()
    assert header[1] == 0 and header[2] == 0, "the last CTA reset the ticket and the counter"
    ug.grid_scan(dev_conteos, inicios, ws, p)
    assert ug.grid_status(ws) == 0
    assert np.array_equal(to_u32(inicios), oracle_lib.exclusive_scan(conteos))


def test_scatter_rejects_cell_out_of_range(ug):
    n, dims = 5000, (8, 8, 8)
    p = ug.make_params(n, dims, (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    celda = torch.randint(0, 512, (n,), dtype=torch.int32, device="cuda")
    celda[1234] = 512                                   # one past the last cell
    counts = torch.bincount(celda.clamp(max=511).long(), minlength=512)
    inicios = torch.zeros(513, dtype=torch.int32, device="cuda")
    inicios[1:] = counts.cumsum(0).int()
    cursor = torch.zeros(512, dtype=torch.int32, device="cuda")
    ordenado = torch.full((n + 64,), -1, dtype=torch.int32, device="cuda")   # 64 guard entries
    ug.grid_scatter(celda, inicios, cursor, ordenado, ws, p)
    assert ug.grid_status(ws) == EBOUNDS
    assert (ordenado[n:] == -1).all(), "nothing written past the end"
    assert ug.grid_status(ws) == 0, "the status word is cleared once read"


def test_reorder_rejects_index_out_of_range(ug):
    n = 3000
    p = ug.make_params(n, (4, 4, 4), (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    origen = torch.randn(n, 8, device="cuda")
    ordenado = torch.randperm(n, device="cuda").int()
    ordenado[17] = n + 5
    destino = torch.zeros(n, 8, device="cuda")
    ug.grid_reorder(ordenado, origen, destino, ws, p)
    assert ug.grid_status(ws) == EBOUNDS
    assert (destino[17] == 0).all(), "the bad record is skipped"
    ok = torch.arange(n, device="cuda") != 17
    assert torch.equal(destino[ok], origen[ordenado[ok].long()])


def test_stable_sort_rejects_inconsistent_starts(ug):
    n, dims = 4000, (10, 10, 10)
    p = ug.make_params(n, dims, (0, 0, 0), 1.0)
    ws = torch.zeros(ug.grid_workspace_bytes(p, ug.GRID_STABLE), dtype=torch.uint8, device="cuda")
    celda = torch.randint(0, 1000, (n,), dtype=torch.int32, device="cuda")
    counts = torch.bincount(celda.long(), minlength=1000)
    inicios = torch.zeros(1001, dtype=torch.int32, device="cuda")
    inicios[1:] = counts.cumsum(0).int()
    inicios[500] = n + 100                               # a start past the end
    cursor = torch.zeros(1000, dtype=torch.int32, device="cuda")
    ordenado = torch.full((n + 64,), -1, dtype=torch.int32, device="cuda")
    ug.grid_scatter(celda, inicios, cursor, ordenado, ws, p, flags=ug.GRID_STABLE)
    assert ug.grid_status(ws) == EBOUNDS
    assert (ordenado[n:] == -1).all()


def test_gpu_still_usable_after_faults(ug, oracle_lib):
    s = scenes.SCENES["tiny"]
    rows = s.particles()
    p = ug.make_params(s.n, s.dims, s.origin, s.cell_size)
    b = ug.GridBuffers.allocate(p)
    b.build(torch.from_numpy(rows).cuda(), p)
    assert ug.grid_status(b.ws) == 0
    assert np.array_equal(to_u32(b.inicios), oracle_lib.build(rows, s.dims, s.origin, s.cell_size)["inicios"])


# A grid barrier's arrival target is raised by the header's bar_extra word
# (word 8).  With it set every CTA still arrives, so all data is written
# before anyone reads it, but no wait ever sees its target: each runs out
# after its one-second limit and the build reports the timeout.  The last
# CTA to leave still resets the barrier words, and the next build with the
# word back at zero is exact.
BAR_EXIT, BAR_EXTRA, BAR_COUNT = 5, 8, 32
BARRIER_SCENES = [
    # (particles, sides, flags): the plan grid_build picks for each
    (40_000, (64, 64, 64), 0),              # sparse: one grid barrier
    (40_000, (64, 64, 64), 1),              # sparse, stable
    (40_000, (16, 16, 16), 0),              # bucketed: two grid barriers
    (40_000, (16, 16, 16), 1),              # bucketed, stable
    (400_000, (512, 512, 257), 0),          # more than 8192 buckets: the fused build
]


@pytest.mark.parametrize("n,dims,flags", BARRIER_SCENES)
def test_grid_barrier_waits_time_out_and_workspace_recovers(ug, oracle_lib, n, dims, flags):
    from gpu_helpers import assert_matches_oracle

    cs = np.float32(0.25)
    rng = np.random.default_rng(n + dims[0] + flags)
    rows = np.zeros((n, 8), np.float32)
    rows[:, :3] = (rng.random((n, 3)) * np.array(dims) * float(cs)).astype(np.float32)
    rows[:, 3:] = rng.random((n, 5)).astype(np.float32)
    p = ug.make_params(n, dims, (0, 0, 0), cs)
    b = ug.GridBuffers.allocate(p, flags)
    origen = torch.from_numpy(rows).cuda()
    words = b.ws.view(torch.int32)
    words[BAR_EXTRA] = 1
    b.build(origen, p, flags)
    assert ug.grid_status(b.ws) == ETIMEOUT
    header = words[:64].cpu().numpy()
    assert header[BAR_COUNT] == 0 and header[BAR_EXIT] == 0, "the last CTA reset the barrier words"
    words[BAR_EXTRA] = 0
    b.build(origen, p, flags)
    got = {
        "status": ug.grid_status(b.ws),
        "conteos": to_u32(b.conteos),
        "celdaDe": to_u32(b.celdaDe),
        "inicios": to_u32(b.inicios),
        "ordenado": to_u32(b.ordenado),
        "destino": b.destino.cpu().numpy(),
    }
    ref = oracle_lib.build(rows, dims, (0, 0, 0), cs)
    assert_matches_oracle(oracle_lib, rows, got, ref, bool(flags))
