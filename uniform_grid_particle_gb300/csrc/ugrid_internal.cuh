// Internal declarations shared by the libugrid translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ugrid.h"

namespace ugrid {

// Bits of grid_ws_header::status.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBounds = 2u;

// Look-back waits give up after this long (the real wait is microseconds).
constexpr unsigned long long kSpinLimitNs = 1000ull * 1000ull * 1000ull;

// Grid geometry as the kernels see it (invCell already rounded on the host).
struct Geometry {
    float origin[3];
    float inv_cell;
    uint32_t dims[3];
};

// ---- scan tiling --------------------------------------------------------
constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;  // four 16-byte vectors per thread
constexpr uint32_t kScanTile = kScanThreads * kScanItems;  // 4096 cells

inline uint64_t scan_tiles(uint64_t cells) { return (cells + kScanTile - 1) / kScanTile; }

// ---- workspace layout ---------------------------------------------------
constexpr size_t kHeaderBytes = 256;
struct WsLayout {
    size_t tile_status;     // u64[tiles]
    size_t stable_queue;    // u32[cells] queue of long segments (GRID_STABLE)
    size_t stable_scratch;  // u32[n] radix-sort scratch (GRID_STABLE)
    size_t total;
};
WsLayout ws_layout(uint64_t n, uint64_t cells, unsigned flags);

// ---- launchers (one per kernel family); all enqueue on `s` --------------
cudaError_t launch_count(const ugrid_particula *parts, uint32_t *conteos, uint32_t *celdaDe,
                         uint32_t n, const Geometry &g, cudaStream_t s);

// inicios = exclusive scan of conteos (C+1 entries).  When zero_input is
// true the kernel also writes zeros over each conteos tile after reading it.
cudaError_t launch_scan(uint32_t *conteos, uint32_t *inicios, uint64_t cells, bool zero_input,
                        grid_ws_header *hdr, unsigned long long *tile_status, cudaStream_t s);

cudaError_t launch_scatter(const uint32_t *celdaDe, const uint32_t *inicios, uint32_t *cursor,
                           uint32_t *ordenado, uint32_t n, uint32_t cells, uint32_t *status,
                           cudaStream_t s);

cudaError_t launch_reorder(const uint32_t *ordenado, const ugrid_particula *origen,
                           ugrid_particula *destino, uint32_t n, uint32_t *status, cudaStream_t s);

// Queue entries needed for cells longer than the register tier (<= cells).
size_t segment_queue_capacity(uint64_t n, uint64_t cells);

cudaError_t launch_segment_sort(const uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                                uint32_t cells, grid_ws_header *hdr, uint32_t *queue,
                                uint32_t *scratch, cudaStream_t s);

// ---- device helpers -----------------------------------------------------
__device__ __forceinline__ void record_status(uint32_t *status, uint32_t bit) {
    atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 16-byte read-only load that does not allocate in L1 (streamed records).
__device__ __forceinline__ uint4 load_nc_na(const uint4 *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte streaming store (evict-first).
__device__ __forceinline__ void store_cs(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace ugrid
