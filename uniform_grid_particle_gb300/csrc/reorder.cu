// a5 — gather reorder of the 32-byte records into cell order.
//
// "Reordenar por celda y la coalescencia de memoria" (§El kernel de
// reordenación): destino[k] = origen[ordenado[k]].  A gather: the writes are
// contiguous and only the reads are scattered (the scatter direction is
// rejected on that page because scattered writes cost more).
//
// Two adjacent threads move one record, 16 bytes each: a warp reads 16 whole
// 32-byte sectors from scattered places and writes 512 contiguous bytes, so
// every sector fetched or written is used in full.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;  // half-records per thread, loads issued before stores

__global__ void __launch_bounds__(kThreads)
reorder_kernel(const uint32_t *__restrict__ ordenado, const uint4 *__restrict__ origen,
               uint4 *__restrict__ destino, uint32_t n, uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kItems) + threadIdx.x;
    uint32_t src[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t h = first + (uint64_t)k * kThreads;  // half-record index
        src[k] = (h >> 1) < n ? __ldg(ordenado + (h >> 1)) : 0u;
    }
    uint4 v[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t h = first + (uint64_t)k * kThreads;
        if ((h >> 1) < n && src[k] < n) v[k] = load_nc_na(origen + 2 * (uint64_t)src[k] + (h & 1));
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const uint64_t h = first + (uint64_t)k * kThreads;
        if ((h >> 1) < n) {
            if (src[k] < n)
                store_cs(destino + h, v[k]);
            else if ((h & 1) == 0)
                record_status(status, kStatusBounds);
        }
    }
}

}  // namespace

cudaError_t launch_reorder(const uint32_t *ordenado, const ugrid_particula *origen,
                           ugrid_particula *destino, uint32_t n, uint32_t *status, cudaStream_t s,
                           bool pdl) {
    if (n == 0) return cudaSuccess;
    const uint64_t halves = 2ull * n;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((halves + per_block - 1) / per_block);
    return launch(reorder_kernel, blocks, kThreads, 0, s, pdl, ordenado,
                  reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino), n,
                  status);
}

}  // namespace ugrid
