"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare it with the CPU oracle under the matching rules.

Matching rules: celdaDe, conteos and inicios bit-exact; ordenado and the
reordered records bit-exact after sorting each cell's segment by particle
index (order inside a cell depends on scheduling); in stable mode bit-exact
with no canonicalisation.
"""
from __future__ import annotations

import numpy as np
import torch


def to_u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def gpu_build(ug, rows: np.ndarray, dims, origin, cs, flags: int = 0, bufs=None, params=None):
    p = params or ug.make_params(rows.shape[0], dims, origin, cs)
    b = bufs or ug.GridBuffers.allocate(p, flags)
    origen = torch.from_numpy(np.ascontiguousarray(rows)).cuda()
    b.build(origen, p, flags)
    status = ug.grid_status(b.ws)
    return {
        "status": status,
        "conteos": to_u32(b.conteos),
        "celdaDe": to_u32(b.celdaDe),
        "inicios": to_u32(b.inicios),
        "ordenado": to_u32(b.ordenado),
        "destino": b.destino.cpu().numpy(),
    }


def assert_matches_oracle(o, rows, got, ref, stable: bool) -> None:
    assert got["status"] == 0, f"device status {got['status']}"
    n = rows.shape[0]
    assert np.array_equal(got["celdaDe"], ref["celdaDe"]), _first_diff(got["celdaDe"], ref["celdaDe"], "celdaDe")
    assert np.array_equal(got["conteos"], ref["conteos"]), _first_diff(got["conteos"], ref["conteos"], "conteos")
    assert np.array_equal(got["inicios"], ref["inicios"]), _first_diff(got["inicios"], ref["inicios"], "inicios")
    ordenado = got["ordenado"]
    # the reordered records are exactly the gathered origen records
    assert np.array_equal(got["destino"].view(np.uint32), rows.view(np.uint32)[ordenado]), "destino != origen[ordenado]"
    if stable:
        assert np.array_equal(ordenado, ref["ordenado"]), _first_diff(ordenado, ref["ordenado"], "ordenado (stable)")
        assert np.array_equal(got["destino"].view(np.uint32), ref["destino"].view(np.uint32))
    else:
        canon = o.canonicalise(got["inicios"], ordenado)
        assert np.array_equal(canon, ref["ordenado"]), _first_diff(canon, ref["ordenado"], "canonical ordenado")
        canon_dest = o.reorder(canon, rows)
        assert np.array_equal(canon_dest.view(np.uint32), ref["destino"].view(np.uint32))
    assert ordenado.size == n


def _first_diff(a, b, name) -> str:
    if a.shape != b.shape:
        return f"{name}: shape {a.shape} vs {b.shape}"
    idx = np.nonzero(a != b)[0]
    if idx.size == 0:
        return f"{name}: equal"
    i = int(idx[0])
    return f"{name}: {idx.size} mismatches, first at {i}: gpu {a[i]} oracle {b[i]}"


def special_rows(dims, origin, cs, seed: int = 0, n: int = 20000) -> np.ndarray:
    """Positions on and next to every cell face, the domain edges, far outside,
    and NaN / infinities: the cases where an FMA or a wrong clamp would show."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    rows = np.zeros((n, 8), dtype=np.float32)
    for d in range(3):
        k = rng.integers(-3, dims[d] + 3, n)
        face = (np.float64(origin[d]) + k * np.float64(cs)).astype(f32)
        step = rng.integers(-2, 3, n)
        v = face.copy()
        for s in (-2, -1, 1, 2):
            sel = step == s
            towards = np.where(s > 0, np.inf, -np.inf).astype(f32)
            w = v[sel]
            for _ in range(abs(s)):
                w = np.nextafter(w, towards)
            v[sel] = w
        rows[:, d] = v
    special = np.array([np.nan, np.inf, -np.inf, 1e30, -1e30, 0.0, -0.0], dtype=f32)
    pick = rng.random((n, 3)) < 0.02
    rows[:, :3][pick] = special[rng.integers(0, special.size, pick.sum())]
    rows[:, 3] = rng.random(n).astype(f32)
    rows[:, 7] = np.arange(n, dtype=f32)
    return rows
