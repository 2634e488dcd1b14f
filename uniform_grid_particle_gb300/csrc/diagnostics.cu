// Overflow diagnostics of a built grid.
//
// "Contar partículas por celda" (§Detectar el desbordamiento sin salir de la
// GPU): with a fixed capacity per cell, particles beyond it would be lost
// silently; the page measures the largest occupancy (maxPorCelda, an atomicMax
// of previo + 1 while counting) and the number of particles that arrived
// over the capacity (desbordes), and reads them back rarely.  Once the count
// is done those two numbers are fixed by the histogram: maxPorCelda is the
// largest count and desbordes is the sum over cells of max(0, count -
// capacity).  This kernel computes them in one pass over conteos, so the
// build itself carries no extra atomics (the page advises keeping the
// diagnostic variant out of the production pipeline).
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads)
diagnostics_kernel(const uint32_t *__restrict__ conteos, uint64_t cells, uint32_t capacidad,
                   uint32_t *diag) {
    __shared__ uint32_t s_most[kWarps], s_over[kWarps];
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    const uint64_t first = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    uint32_t most = 0, over = 0;
    const uint64_t quads = cells / 4;
    const uint4 *c4 = reinterpret_cast<const uint4 *>(conteos);
#pragma unroll 4
    for (uint64_t q = first; q < quads; q += stride) {
        const uint4 v = c4[q];
        most = max(max(most, max(v.x, v.y)), max(v.z, v.w));
        over += (v.x > capacidad ? v.x - capacidad : 0u) + (v.y > capacidad ? v.y - capacidad : 0u) +
                (v.z > capacidad ? v.z - capacidad : 0u) + (v.w > capacidad ? v.w - capacidad : 0u);
    }
    for (uint64_t c = quads * 4 + first; c < cells; c += stride) {
        const uint32_t v = conteos[c];
        most = max(most, v);
        over += v > capacidad ? v - capacidad : 0u;
    }
    // Warp, then block: one pair of atomics per block, so the two words are
    // not a queue of thousands of same-address atomics.
    most = __reduce_max_sync(0xffffffffu, most);
    over = __reduce_add_sync(0xffffffffu, over);
    if (lane_id() == 0) {
        s_most[threadIdx.x >> 5] = most;
        s_over[threadIdx.x >> 5] = over;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        most = threadIdx.x < kWarps ? s_most[threadIdx.x] : 0u;
        over = threadIdx.x < kWarps ? s_over[threadIdx.x] : 0u;
        most = __reduce_max_sync(0xffffffffu, most);
        over = __reduce_add_sync(0xffffffffu, over);
        if (threadIdx.x == 0) {
            if (most) atomicMax(diag, most);
            if (over) atomicAdd(diag + 1, over);
        }
    }
}

}  // namespace

cudaError_t launch_diagnostics(const uint32_t *conteos, uint64_t cells, uint32_t capacidad,
                               uint32_t *diag, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(diag, 0, 2 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    int device = 0, sms = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
        return e;
    // Two blocks per SM at most: every thread has a few 16-byte loads in flight.
    const uint64_t want = (cells / 4 + kThreads - 1) / kThreads;
    const unsigned blocks = (unsigned)(want < 1 ? 1 : (want < (uint64_t)sms * 2 ? want : (uint64_t)sms * 2));
    return launch(diagnostics_kernel, blocks, kThreads, 0, s, false, conteos, cells, capacidad, diag);
}

}  // namespace ugrid
