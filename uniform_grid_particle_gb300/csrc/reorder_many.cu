// Gather reorder of several particle arrays with one index read.
//
// "Reordenar por celda y la coalescencia de memoria" (§El kernel de
// reordenación): when the particle state lives in several buffers — the hot
// Cinematica and the cold Aspecto of "El estado de las partículas en storage
// buffers" (§AoS o SoA) — the same ordenado is applied to all of them, and one
// kernel that reads ordenado[k] once for every pair is better than one kernel
// per pair.  For every array a and every k < N:
//     destino_a[k] = origen_a[ordenado[k]]   (records of record_bytes_a bytes)
//
// Each record is cut into 16-byte pieces and the pieces of all arrays for one
// k are handed to adjacent threads, which read the same ordenado[k] (one
// transaction) and write each array's records contiguously.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;  // pieces per thread, loads issued before stores

__global__ void __launch_bounds__(kThreads)
reorder_many_kernel(const uint32_t *__restrict__ ordenado, const __grid_constant__ ManyArrays m, uint32_t n,
                    uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t pieces = (uint64_t)n * m.per_record;
    const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kItems) + threadIdx.x;
    uint32_t src[kItems], arr[kItems], piece[kItems];
    uint64_t rec[kItems];
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
        const uint64_t g = first + (uint64_t)t * kThreads;
        rec[t] = g / m.per_record;
        uint32_t j = (uint32_t)(g - rec[t] * m.per_record);
        uint32_t a = 0;
        while (a + 1 < m.count && j >= m.first[a + 1]) ++a;
        arr[t] = a;
        piece[t] = j - m.first[a];
        src[t] = g < pieces ? __ldg(ordenado + rec[t]) : 0u;
    }
    uint4 v[kItems];
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
        const uint64_t g = first + (uint64_t)t * kThreads;
        if (g < pieces && src[t] < n)
            v[t] = load_nc_na(m.src[arr[t]] + (uint64_t)src[t] * m.pieces[arr[t]] + piece[t]);
    }
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
        const uint64_t g = first + (uint64_t)t * kThreads;
        if (g < pieces) {
            if (src[t] < n)
                store_cs(m.dst[arr[t]] + rec[t] * m.pieces[arr[t]] + piece[t], v[t]);
            else if (m.first[arr[t]] + piece[t] == 0)
                record_status(status, kStatusBounds);
        }
    }
}

}  // namespace

cudaError_t launch_reorder_many(const uint32_t *ordenado, const ManyArrays &m, uint32_t n,
                                uint32_t *status, cudaStream_t s, bool pdl) {
    if (n == 0) return cudaSuccess;
    const uint64_t pieces = (uint64_t)n * m.per_record;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((pieces + per_block - 1) / per_block);
    return launch(reorder_many_kernel, blocks, kThreads, 0, s, pdl, ordenado, m, n, status);
}

}  // namespace ugrid
