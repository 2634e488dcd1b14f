// a2 — per-particle cell index and histogram.
//
// "Contar partículas por celda" (§El kernel): the cell of particle i is saved
// in celdaDe[i] and conteos[c] is incremented atomically; the clamp lives in
// the cell-index helper.  §La contención de las celdas densas: when the
// particles of one SIMD group share a cell they add to its counter once
// (here: __match_any_sync, then the lowest lane of each group adds the group
// size).  The grouping runs only when some lane holds the same cell as the
// lane before it — particles already in cell order, or clustered ones; for
// scattered particles it would cost more than it saves.  "Reordenar por celda…" (§El orden de las celdas): c = x + y*GX +
// z*GX*GY.
//
// Each thread reads only the first 16 bytes of its 32-byte record (pos and
// vida) with one vector load; the counters stay in L2.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;  // particles per thread, loads issued before any use

template <bool kAggregate>
__global__ void __launch_bounds__(kThreads)
count_kernel(const uint4 *__restrict__ parts, uint32_t *__restrict__ conteos,
             uint32_t *__restrict__ celdaDe, uint32_t n, Geometry g) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kItems) + threadIdx.x;
    uint4 rec[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t i = first + (uint64_t)k * kThreads;
        if (i < n) rec[k] = load_nc_na(parts + 2 * i);  // bytes 0..15: pos, vida
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t i = first + (uint64_t)k * kThreads;
        const bool valid = i < n;
        const uint32_t c = valid ? cell_of(rec[k], g) : 0u;
        if (valid) celdaDe[i] = c;
        if (kAggregate && warp_has_adjacent_duplicates(valid, c)) {
            const uint32_t active = __ballot_sync(0xffffffffu, valid);
            if (valid) {
                const uint32_t peers = __match_any_sync(active, c);
                if (lane_id() == (uint32_t)(__ffs(peers) - 1)) atomicAdd(conteos + c, __popc(peers));
            }
        } else if (valid) {
            atomicAdd(conteos + c, 1u);
        }
    }
}

}  // namespace

cudaError_t launch_count(const ugrid_particula *parts, uint32_t *conteos, uint32_t *celdaDe,
                         uint32_t n, const Geometry &g, cudaStream_t s, bool pdl) {
    if (n == 0) return cudaSuccess;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((n + per_block - 1) / per_block);
    return launch(count_kernel<true>, blocks, kThreads, 0, s, pdl,
                  reinterpret_cast<const uint4 *>(parts), conteos, celdaDe, n, g);
}

}  // namespace ugrid
