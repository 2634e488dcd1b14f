// Internal declarations shared by the libugrid translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ugrid.h"

namespace ugrid {

// Bits of grid_ws_header::status.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBounds = 2u;

// Look-back waits give up after this long (the real wait is microseconds).
constexpr unsigned long long kSpinLimitNs = 1000ull * 1000ull * 1000ull;

// Grid geometry as the kernels see it (invCell already rounded on the host).
// Cell orders as the kernels see them: the public GRID_ORDER_MORTON splits
// into the cubic case (three equal sides, at most 2^10 each: a shift-and-mask
// spread) and the general one (a bit deposit through per-axis masks).
constexpr uint32_t kOrderLinear = 0u;
constexpr uint32_t kOrderMorton = 1u;
constexpr uint32_t kOrderMortonCubic = 2u;

struct Geometry {
    float origin[3];
    float inv_cell;
    uint32_t dims[3];
    uint32_t order;
    uint32_t mask[3];  // Morton: the code bits each axis's bits go to, low to high
};

// ---- scan tiling --------------------------------------------------------
constexpr int kScanThreads = 512;
constexpr int kScanItems = 16;  // four 16-byte vectors per thread
constexpr uint32_t kScanTile = kScanThreads * kScanItems;  // 8192 cells

inline uint64_t scan_tiles(uint64_t cells) { return (cells + kScanTile - 1) / kScanTile; }
// u64 words from one tile's look-back word to the next in a workspace: one
// 128-byte line each, so that the polls of all tiles spread over many L2
// slices instead of hammering the few lines a dense array would take.
constexpr uint32_t kLookStride = 16;

// ---- workspace layout ---------------------------------------------------
constexpr size_t kHeaderBytes = 256;
constexpr uint32_t kFusedMaxCtas = 4096;  // bound on the fused build's grid
// The bucketed build groups the cells into buckets of `width` consecutive
// cells.  A bucket's counters, and a CTA's counters of all buckets, each fill
// one CTA's 32 KB table, so both are capped at 8192; a bucket holding more
// than kBucketCap particles sends the whole build down the atomic path.
constexpr uint32_t kBucketMaxCells = 8192;
constexpr uint32_t kBucketMaxCount = 8192;
constexpr uint32_t kBucketCap = 4096;   // particles one CTA places in shared memory
constexpr uint32_t kBucketAvg = 3300;   // particles per bucket aimed at (uniform scenes stay far below the cap)
constexpr uint32_t kBucketLanes = 8;    // counters per bucket, so that few CTAs add to the same word
struct BucketPlan {
    uint32_t width;              // cells per bucket, a multiple of 4
    uint32_t buckets;            // 0: the bucketed build is not used
    unsigned long long magic;    // ceil(2^64 / width): bucket = umulhi64(cell, magic)
};
// A whole number of buckets per CTA of the launch (`ctas`), each holding
// about kBucketAvg particles of a uniform scene, with at most kBucketMaxCells
// cells per bucket and kBucketMaxCount buckets.
inline BucketPlan bucket_plan(uint64_t n, uint64_t cells, uint32_t ctas) {
    BucketPlan p{0u, 0u, 0ull};
    if (n == 0 || cells == 0 || ctas == 0) return p;
    const uint64_t per_cta = (n + (uint64_t)ctas * kBucketAvg - 1) / ((uint64_t)ctas * kBucketAvg);
    uint64_t b = (uint64_t)ctas * per_cta;
    uint64_t w = (cells + b - 1) / b;
    w = (w + 3) & ~3ull;
    if (w > kBucketMaxCells) w = kBucketMaxCells;
    b = (cells + w - 1) / w;
    if (b > kBucketMaxCount) return p;
    p.width = (uint32_t)w;
    p.buckets = (uint32_t)b;
    p.magic = ~0ull / w + 1ull;  // w >= 4, so this is ceil(2^64 / w)
    return p;
}

struct WsLayout {
    size_t tile_status;     // u64[tiles * kLookStride]: one look-back word per 128-byte line
    size_t chunk_sums;      // u32[kFusedMaxCtas] per-CTA cell-chunk totals (fused build)
    size_t slots;           // u32[n] slot of each particle in its cell (fused build)
    size_t counts;          // u32[cells] counters of the fused build, zero between builds
    size_t bucket_total;    // u32[kBucketMaxCount][kBucketLanes] particles per bucket and lane, zero between builds
    size_t bucket_base;     // u32[kBucketMaxCount] first position of each bucket
    size_t pairs;           // u32x2[n] (cell, particle) grouped by bucket
    size_t stable_queue;    // u32[cells] queue of long segments (GRID_STABLE)
    size_t stable_scratch;  // u32[n] radix-sort scratch (GRID_STABLE)
    size_t total;
};
WsLayout ws_layout(uint64_t n, uint64_t cells, unsigned flags);

// ---- launch helper --------------------------------------------------------
// With `pdl` the kernel may be launched while the previous kernel on the
// stream is still running (programmatic dependent launch); every kernel
// starts with grid_dependency_wait() before it touches memory the previous
// kernel wrote, so results are the same either way.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                   cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- launchers (one per kernel family); all enqueue on `s` --------------
cudaError_t launch_count(const ugrid_particula *parts, uint32_t *conteos, uint32_t *celdaDe,
                         uint32_t n, const Geometry &g, cudaStream_t s, bool pdl);

// inicios = exclusive scan of conteos (C+1 entries).  When zero_input is
// true the kernel also writes zeros over each conteos tile after reading it.
cudaError_t launch_scan(uint32_t *conteos, uint32_t *inicios, uint64_t cells, bool zero_input,
                        grid_ws_header *hdr, unsigned long long *tile_status, uint32_t stride, cudaStream_t s,
                        bool pdl);

cudaError_t launch_scatter(const uint32_t *celdaDe, const uint32_t *inicios, uint32_t *cursor,
                           uint32_t *ordenado, uint32_t n, uint32_t cells, uint32_t *status,
                           cudaStream_t s, bool pdl);

// origen described to the tensor memory accelerator as n rows of eight u32
// words, with a box of one whole row (the form a tile::gather4 copy reads).
cudaError_t record_tensor_map(const ugrid_particula *origen, uint32_t n, CUtensorMap *map);
// The same for any array of `rows` rows of row_bytes bytes (a multiple of 16,
// at most 1024), read as u32 words.
cudaError_t rows_tensor_map(const void *base, uint32_t row_bytes, uint32_t rows, CUtensorMap *map);

cudaError_t launch_reorder(const uint32_t *ordenado, const ugrid_particula *origen,
                           ugrid_particula *destino, uint32_t n, uint32_t *status, cudaStream_t s,
                           bool pdl);

// The whole build in one cooperative launch (see build_fused.cu).
// Returns cudaErrorNotSupported when the device cannot run it, so the caller
// can fall back to one launch per phase.
cudaError_t launch_build_fused(const ugrid_particula *origen, ugrid_particula *destino,
                               uint32_t *conteos, uint32_t *celdaDe, uint32_t *inicios,
                               uint32_t *ordenado, uint32_t n, uint64_t cells, const Geometry &g,
                               grid_ws_header *hdr, uint32_t *chunk_sums, uint32_t *slots,
                               uint32_t *counts, bool stable, uint32_t *queue,
                               uint32_t queue_capacity, uint32_t *sort_scratch, cudaStream_t s);
cudaError_t launch_build_bucketed(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                  uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                                  uint64_t cells, const Geometry &g, grid_ws_header *hdr, uint32_t *chunk_sums,
                                  uint32_t *slots, uint32_t *counts, uint32_t *total, uint32_t *base,
                                  uint32_t *pairs, bool stable, uint32_t *queue, uint32_t queue_capacity,
                                  uint32_t *sort_scratch, cudaStream_t s);

// The non-stable build of a small scene on one thread-block cluster of up to
// kClusterMaxCtas CTAs sharing its cell table in distributed shared memory
// (see build_cluster.cu).  Returns cudaErrorNotSupported, having launched
// nothing, when the device runs no cluster large enough for the scene.
constexpr uint32_t kClusterMaxCtas = 16;
// (measured: at 30,000 particles the cluster build and the bucketed build
// take the same time, at 65,536 the bucketed build is faster)
constexpr uint32_t kClusterMaxParticles = 32768;
constexpr uint32_t kClusterMaxCells = 131072;
cudaError_t launch_build_cluster(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                 uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n, uint32_t cells,
                                 const Geometry &g, cudaStream_t s);

// The whole build in one CTA, for scenes of at most kSmallMaxParticles
// particles on at most kSmallMaxCells cells (see build_small.cu).
constexpr uint32_t kSmallMaxParticles = 8192;
constexpr uint32_t kSmallMaxCells = 8192;
cudaError_t launch_build_small(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                               uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                               uint32_t cells, const Geometry &g, bool stable, cudaStream_t s);

// The sparse build: at most this many particles per CTA of its launch
// (measured: with more, its plain-load gather and its phase 1 make it slower
// than the bucketed build).
constexpr uint32_t kSparseMaxParticlesPerCta = 1024;
// grid_build takes the sparse build when there are at least this many cells
// per particle.
constexpr uint64_t kSparseCellsPerParticle = 4;
// The build for sparse grids, one cooperative launch with one grid barrier
// (see build_sparse.cu).  Its table of per-CTA bucket offsets lives in the
// fused build's counter array `counts` (the kernel marks it not clean).
// Returns cudaErrorNotSupported, having launched nothing, when a CTA's
// particles would not fit (n > grid * kSparseMaxParticlesPerCta) or the table
// would not fit in `cells` words.
cudaError_t launch_build_sparse(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n, uint64_t cells,
                                const Geometry &g, grid_ws_header *hdr, uint32_t *counts, uint32_t *pairs,
                                bool stable, uint32_t *sort_scratch, cudaStream_t s);

// Several arrays gathered with one ordenado (grid_reorder_many).
constexpr int kMaxArrays = 4;
struct ManyArrays {
    const uint4 *src[kMaxArrays];
    uint4 *dst[kMaxArrays];
    uint32_t pieces[kMaxArrays];     // 16-byte pieces per record of each array
    uint32_t first[kMaxArrays + 1];  // running sum of pieces: array a owns [first[a], first[a+1])
    uint32_t count;                  // arrays in use
    uint32_t per_record;             // pieces of all arrays for one record
};
cudaError_t launch_reorder_many(const uint32_t *ordenado, const ManyArrays &m, uint32_t n,
                                uint32_t *status, cudaStream_t s, bool pdl);

// rho[k] = neighbour density of the particle at cell-order position k (parts =
// destino when ordenado is null, else origen read through ordenado).
cudaError_t launch_density(const ugrid_particula *parts, const uint32_t *ordenado,
                           const uint32_t *inicios, const Geometry &g, float h, uint32_t n,
                           float *rho, uint32_t *status, cudaStream_t s);

// diag[0] = max over cells of conteos, diag[1] = sum of max(0, conteos - capacidad).
cudaError_t launch_diagnostics(const uint32_t *conteos, uint64_t cells, uint32_t capacidad,
                               uint32_t *diag, cudaStream_t s);

// Queue entries needed for cells longer than the register tier (<= cells).
size_t segment_queue_capacity(uint64_t n, uint64_t cells);

cudaError_t launch_segment_sort(const uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                                uint32_t cells, grid_ws_header *hdr, uint32_t *queue,
                                uint32_t *scratch, cudaStream_t s, bool pdl);

// ---- device helpers -----------------------------------------------------
__device__ __forceinline__ void record_status(uint32_t *status, uint32_t bit) {
    atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Clamped cell coordinate along one axis ("Contar partículas por celda",
// §El kernel: the range guard lives in the cell-index helper):
// floor((p - o) * invCell) in fp32, round-to-nearest subtraction and
// multiplication (never contracted), saturated to [0, dim - 1].  `f >= 0` is
// false for NaN, so NaN goes to 0; the float-to-unsigned conversion saturates
// +inf and huge values, and the min() brings them to dim - 1.
__device__ __forceinline__ uint32_t axis_coord(float p, float o, float inv, uint32_t dim) {
    const float f = floorf(__fmul_rn(__fsub_rn(p, o), inv));
    return f >= 0.0f ? min(__float2uint_rz(f), dim - 1u) : 0u;
}

// Bit i of the low ten bits of v moved to bit 3i (the classic halving spread:
// each step moves the upper half of every group up by twice its distance).
__device__ __forceinline__ uint32_t spread3(uint32_t v) {
    v &= 0x3ffu;
    v = (v | (v << 16)) & 0x030000ffu;
    v = (v | (v << 8)) & 0x0300f00fu;
    v = (v | (v << 4)) & 0x030c30c3u;
    v = (v | (v << 2)) & 0x09249249u;
    return v;
}

// The low bits of v placed, in order, at the set bits of mask.
__device__ __forceinline__ uint32_t deposit(uint32_t v, uint32_t mask) {
    uint32_t out = 0u;
    for (uint32_t m = mask; m != 0u; m &= m - 1u, v >>= 1)
        if (v & 1u) out |= m & (0u - m);
    return out;
}

// Index of cell (x, y, z) in the grid's order ("Reordenar por celda…", §El
// orden de las celdas): linear x + y*GX + z*GX*GY, or the Z-curve interleave.
__device__ __forceinline__ uint32_t cell_at(uint32_t x, uint32_t y, uint32_t z, const Geometry &g) {
    if (g.order == kOrderLinear) return x + g.dims[0] * (y + g.dims[1] * z);
    if (g.order == kOrderMortonCubic) return spread3(x) | (spread3(y) << 1) | (spread3(z) << 2);
    return deposit(x, g.mask[0]) | deposit(y, g.mask[1]) | deposit(z, g.mask[2]);
}

// Cell index of the position in the first 16 bytes of a record.
__device__ __forceinline__ uint32_t cell_of(const uint4 &rec, const Geometry &g) {
    const uint32_t x = axis_coord(__uint_as_float(rec.x), g.origin[0], g.inv_cell, g.dims[0]);
    const uint32_t y = axis_coord(__uint_as_float(rec.y), g.origin[1], g.inv_cell, g.dims[1]);
    const uint32_t z = axis_coord(__uint_as_float(rec.z), g.origin[2], g.inv_cell, g.dims[2]);
    return cell_at(x, y, z, g);
}

// True (for the whole warp) when some valid lane holds the same key as the
// valid lane just below it: the cheap test that decides whether grouping the
// warp's atomics by key with __match_any_sync is worth it.
__device__ __forceinline__ bool warp_has_adjacent_duplicates(bool valid, uint32_t key) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    const uint32_t below = __shfl_up_sync(0xffffffffu, key, 1);
    const bool dup = valid && lane > 0 && ((active >> (lane - 1)) & 1u) && below == key;
    return __any_sync(0xffffffffu, dup);
}

// Programmatic dependent launch: wait for the previous grid's memory to be
// visible (a no-op when the kernel was launched normally), and let the next
// grid begin launching once every CTA of this one has started.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Shared-memory add of 1 to table[key] for every valid lane; returns the
// value before this lane's add.  Lanes of a warp that share a key are served
// by one atomic of their leader when the cheap adjacent-duplicate test finds
// any, so crowded keys do not serialise.  When the valid lanes are a prefix of
// the warp and their keys do not decrease (input already in cell order), the
// runs of equal keys are found with one ballot: each run's first lane adds
// the run's length.  Otherwise __match_any_sync groups the lanes.
__device__ __forceinline__ uint32_t smem_take(uint32_t *table, bool valid, uint32_t key) {
    if (!warp_has_adjacent_duplicates(valid, key)) return valid ? atomicAdd(&table[key], 1u) : 0u;
    const uint32_t lane = lane_id();
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    const uint32_t below = __shfl_up_sync(0xffffffffu, key, 1);
    const bool prefix = (active & (active + 1u)) == 0u;  // lanes 0..k-1 valid, the rest not
    if (prefix && __all_sync(0xffffffffu, !valid || lane == 0 || below <= key)) {
        const uint32_t heads = __ballot_sync(0xffffffffu, valid && (lane == 0 || below != key));
        const uint32_t upto = lane == 31 ? 0xffffffffu : (2u << lane) - 1u;
        const uint32_t start = 31u - (uint32_t)__clz(heads & upto);
        const uint32_t later = (heads | ~active) & ~upto;  // the next run's head, or the first invalid lane
        const uint32_t end = later ? (uint32_t)(__ffs(later) - 1) : 32u;
        uint32_t first = 0u;
        if (valid && lane == start) first = atomicAdd(&table[key], end - start);
        first = __shfl_sync(0xffffffffu, first, start);
        return valid ? first + (lane - start) : 0u;
    }
    uint32_t first = 0u, peers = 0u;
    if (valid) {
        peers = __match_any_sync(active, key);
        const uint32_t leader = (uint32_t)(__ffs(peers) - 1);
        if (lane == leader) first = atomicAdd(&table[key], (uint32_t)__popc(peers));
        first = __shfl_sync(peers, first, leader);
    }
    return first + (uint32_t)__popc(peers & lanemask_lt());
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

// The bytes [p, p + bytes) fetched into L2 by the bulk copy engine: a hint,
// over the 16-byte aligned part of the range only (the start rounded up and
// the end rounded down), so it never touches a byte outside it.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(p) + 15) & ~(uintptr_t)15;
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes) & ~(uintptr_t)15;
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
}

// 16-byte streaming store (evict-first).
__device__ __forceinline__ void store_cs(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- Tensor memory accelerator: a gather of four 32-byte records ----------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

// The one arrival of a phase, expecting `bytes` from copies (0: none).
__device__ __forceinline__ void mbar_arrive_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Wait for the phase of the given parity to complete; false after 1 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long start = global_ns();
    uint32_t polls = 0;
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((++polls & 63u) == 0 && global_ns() - start > kSpinLimitNs) return false;
    }
}

// Rows r0..r3 of a record tensor map (record_tensor_map) into 128 contiguous
// bytes at dst (128-byte aligned), counted on the mbarrier.
__device__ __forceinline__ void gather4_records(uint32_t dst, const CUtensorMap *map, const int (&r)[4],
                                                uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(0), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(bar)
        : "memory");
}

// Rows of a chunk closer together than this are read with plain 16-byte
// loads, which then share lines and sectors; TMA gathers serve scattered rows.
constexpr uint32_t kClusterRows = 512;

// The span (largest - smallest) of the warp's rows, lane l holding v of them.
__device__ __forceinline__ uint32_t rows_span(const int (&row)[4], uint32_t v) {
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if ((uint32_t)e < v) {
            lo = min(lo, (uint32_t)row[e]);
            hi = max(hi, (uint32_t)row[e]);
        }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    return hi >= lo ? hi - lo : 0u;
}

// One bulk copy of `bytes` (a multiple of 16) from shared memory to global
// memory, then wait until the source has been read.
__device__ __forceinline__ void bulk_store_wait_read(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace ugrid
