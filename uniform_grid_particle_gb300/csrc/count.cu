// a2 — per-particle cell index and histogram.
//
// "Contar partículas por celda" (§El kernel): the cell of particle i is saved
// in celdaDe[i] and conteos[c] is incremented atomically; the clamp lives in
// the cell-index helper.  §La contención de las celdas densas: when the
// particles of one SIMD group share a cell they add to its counter once
// (here: __match_any_sync, then the lowest lane of each group adds the group
// size).  "Reordenar por celda…" (§El orden de las celdas): c = x + y*GX +
// z*GX*GY.
//
// Each thread reads only the first 16 bytes of its 32-byte record (pos and
// vida) with one vector load; the counters stay in L2.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;  // particles per thread, loads issued before any use

// Clamped cell coordinate along one axis: floor((p - o) * invCell) in fp32,
// round-to-nearest subtraction and multiplication (never contracted), then
// saturated to [0, dim - 1].  `f >= 0` is false for NaN, so NaN goes to 0;
// the float-to-unsigned conversion saturates +inf and huge values, and the
// min() brings them to dim - 1.
__device__ __forceinline__ uint32_t axis_coord(float p, float o, float inv, uint32_t dim) {
    const float f = floorf(__fmul_rn(__fsub_rn(p, o), inv));
    return f >= 0.0f ? min(__float2uint_rz(f), dim - 1u) : 0u;
}

__device__ __forceinline__ uint32_t cell_of(const uint4 &rec, const Geometry &g) {
    const uint32_t x = axis_coord(__uint_as_float(rec.x), g.origin[0], g.inv_cell, g.dims[0]);
    const uint32_t y = axis_coord(__uint_as_float(rec.y), g.origin[1], g.inv_cell, g.dims[1]);
    const uint32_t z = axis_coord(__uint_as_float(rec.z), g.origin[2], g.inv_cell, g.dims[2]);
    return x + g.dims[0] * (y + g.dims[1] * z);
}

template <bool kAggregate>
__global__ void __launch_bounds__(kThreads)
count_kernel(const uint4 *__restrict__ parts, uint32_t *__restrict__ conteos,
             uint32_t *__restrict__ celdaDe, uint32_t n, Geometry g) {
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
        if (kAggregate) {
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
                         uint32_t n, const Geometry &g, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const uint64_t per_block = (uint64_t)kThreads * kItems;
    const unsigned blocks = (unsigned)((n + per_block - 1) / per_block);
    count_kernel<true><<<blocks, kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(parts),
                                                   conteos, celdaDe, n, g);
    return cudaGetLastError();
}

}  // namespace ugrid
