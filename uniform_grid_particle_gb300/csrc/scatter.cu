// a4 — cursor scatter into cell-grouped order.
//
// "Construir el índice de la rejilla con un prefix sum" (§La dispersión):
// slot = atomicAdd(&cursor[c], 1); ordenado[inicios[c] + slot] = i, with the
// cursor array being conteos again after a clear.  Particles of one warp that
// share a cell take their slots with one atomic: the lowest lane of each group
// (found with __match_any_sync) adds the group size, and each member's slot is
// the returned base plus its rank among the group's lower lanes.  The order
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
    const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kItems) + threadIdx.x;
    uint32_t cell[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t i = first + (uint64_t)k * kThreads;
        cell[k] = i < n ? celdaDe[i] : 0u;
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t i = first + (uint64_t)k * kThreads;
        bool valid = i < n;
        const uint32_t c = cell[k];
        if (valid && c >= cells) {
            record_status(status, kStatusBounds);
            valid = false;
        }
        uint32_t pos = 0;
        if (kAggregate) {
            const uint32_t active = __ballot_sync(0xffffffffu, valid);
            if (valid) {
                const uint32_t peers = __match_any_sync(active, c);
                const uint32_t leader = (uint32_t)(__ffs(peers) - 1);
                uint32_t base = 0;
                if (lane_id() == leader) base = __ldg(inicios + c) + atomicAdd(cursor + c, __popc(peers));
                base = __shfl_sync(peers, base, leader);
                pos = base + __popc(peers & lanemask_lt());
            }
        } else if (valid) {
            pos = __ldg(inicios + c) + atomicAdd(cursor + c, 1u);
        }
        if (valid) {
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
                           cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((n + per_block - 1) / per_block);
    scatter_kernel<true><<<blocks, kThreads, 0, s>>>(celdaDe, inicios, cursor, ordenado, n, cells,
                                                     status);
    return cudaGetLastError();
}

}  // namespace ugrid
