"""grid_scan_noalloc: the scan for callers that cannot allocate device memory.

Engines that own every device buffer, or per-frame steps that cannot risk a
cudaMalloc stalling the device, cannot hand grid_scan a workspace.  This entry
point keeps the scan's scratch in a fixed array inside the library; these
tests check that it gives exactly grid_scan's result, call after call, and
that it refuses inputs larger than that array serves.  The file sorts last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

ERANGE = 5
MAX_CELLS = 4096 * 8192


@pytest.fixture(scope="module")
def ug():
    from uniform_grid_particle_gb300 import build, ugrid

    build.build()
    return ugrid


def test_oversize_is_refused_before_any_cuda_call(ug):
    p = ug.make_params(10, (MAX_CELLS // 4096 + 1, 4096, 1), (0, 0, 0), 1.0)
    fake = 0x7F0000000000
    code = ug.lib().grid_scan_noalloc(fake, fake + (1 << 33), ctypes.byref(p), None)
    assert code == ERANGE
    assert "fixed scratch" in ug.error_string(code)


@pytest.mark.gpu
def test_matches_grid_scan_on_two_calls_in_a_row(ug, oracle_lib):
    rng = np.random.default_rng(2024)
    cases = [
        ((128, 128, 128), rng.poisson(0.477, 128 ** 3).astype(np.uint32)),    # headline-like counts
        ((61, 33, 17), rng.integers(0, 40, 61 * 33 * 17, dtype=np.uint32)),  # ragged, larger counts
    ]
    outs = []
    for dims, counts in cases:   # two calls in a row, nothing in between
        C = dims[0] * dims[1] * dims[2]
        p = ug.make_params(int(counts.sum()), dims, (0, 0, 0), 1.0)
        conteos = torch.from_numpy(counts.view(np.int32)).cuda()
        inicios = torch.full((C + 1,), -1, dtype=torch.int32, device="cuda")
        ug.grid_scan_noalloc(conteos, inicios, p)
        outs.append((dims, counts, conteos, inicios, p))
    torch.cuda.synchronize()
    for dims, counts, conteos, inicios, p in outs:
        C = counts.size
        ws = torch.zeros(ug.grid_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
        ref = torch.empty(C + 1, dtype=torch.int32, device="cuda")
        ug.grid_scan(conteos, ref, ws, p)
        assert ug.grid_status(ws) == 0
        got = inicios.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, ref.cpu().numpy().view(np.uint32)), f"differs from grid_scan at {dims}"
        assert np.array_equal(got, oracle_lib.exclusive_scan(counts))
