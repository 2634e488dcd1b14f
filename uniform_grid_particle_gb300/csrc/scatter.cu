// a4 — cursor scatter into cell-grouped order.
//
// "Construir el índice de la rejilla con un prefix sum" (§La dispersión):
// slot = atomicAdd(&cursor[c], 1); ordenado[inicios[c] + slot] = i, with the
// cursor array being conteos again after a clear.  Particles of one warp that
// share a cell take their slots with one atomic: the lowest lane of each group
// (found with __match_any_sync) adds the group size, and each member's slot is
// the returned base plus its rank among the group's lower lanes.  The grouping
// runs only when some lane holds the same cell as the lane before it.  The order
// inside a cell still depends on scheduling (§El orden dentro de la celda).
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;

template <bool kAggregate>
__global__ void __launch_bounds__(kThreads)
scatter_kernel(const uint32_t *__restrict__ celdaDe, const uint32_t *__restrict__ inicios,
               uint32_t *__restrict__ cursor, uint32_t *__restrict__ ordenado, uint32_t n,
               uint32_t cells, uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kItems) + threadIdx.x;
    const uint32_t lane = lane_id();
    uint32_t cell[kItems];
    bool valid[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t i = first + (uint64_t)k * kThreads;
        valid[k] = i < n;
        cell[k] = valid[k] ? celdaDe[i] : 0u;
    }
    // Claim slots: every item's atomic is issued before any result is used,
    // so the round trips to L2 overlap.
    uint32_t peers[kItems], base[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        if (valid[k] && cell[k] >= cells) {
            record_status(status, kStatusBounds);
            valid[k] = false;
        }
        base[k] = 0;
        // peers = this lane alone unless the warp groups its atomics by cell
        peers[k] = 1u << lane;
        if (kAggregate && warp_has_adjacent_duplicates(valid[k], cell[k])) {
            const uint32_t active = __ballot_sync(0xffffffffu, valid[k]);
            if (valid[k]) peers[k] = __match_any_sync(active, cell[k]);
        }
        if (valid[k] && lane == (uint32_t)(__ffs(peers[k]) - 1))
            base[k] = __ldg(inicios + cell[k]) + atomicAdd(cursor + cell[k], __popc(peers[k]));
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        // Each group's leader holds the group's first slot; members add their
        // rank among the group's lower lanes.
        const uint32_t leader = (uint32_t)(__ffs(peers[k]) - 1);
        const uint32_t pos = __shfl_sync(0xffffffffu, base[k], leader) + __popc(peers[k] & lanemask_lt());
        if (valid[k]) {
            const uint64_t i = first + (uint64_t)k * kThreads;
            if (pos < n)
                ordenado[pos] = (uint32_t)i;
            else
                record_status(status, kStatusBounds);
        }
    }
}

}  // namespace

cudaError_t launch_scatter(const uint32_t *celdaDe, const uint32_t *inicios, uint32_t *cursor,
                           uint32_t *ordenado, uint32_t n, uint32_t cells, uint32_t *status,
                           cudaStream_t s, bool pdl) {
    if (n == 0) return cudaSuccess;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((n + per_block - 1) / per_block);
    return launch(scatter_kernel<true>, blocks, kThreads, 0, s, pdl, celdaDe, inicios, cursor,
                  ordenado, n, cells, status);
}

}  // namespace ugrid
