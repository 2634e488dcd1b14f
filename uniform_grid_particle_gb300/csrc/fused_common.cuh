// Building blocks of the single-launch grid builds: the grid barrier, the
// block scans, and the phases of the atomic counting sort ("Contar partículas
// por celda", "Construir el índice de la rejilla con un prefix sum",
// "Reordenar por celda y la coalescencia de memoria"), written as device
// functions so that the fused build and the bucketed build's fallback run the
// same code.  Every function here is called by all threads of a CTA.
#pragma once

#include "segsort_device.cuh"

namespace ugrid {
namespace fused {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCountItems = 4;    // particles per thread per round
constexpr int kScatterItems = 8;  // particles per thread per round
constexpr int kGatherItems = 4;   // half-records per thread per round
constexpr int kMoveItems = 4;     // half-records per thread per round
constexpr int kScanVecs = 4;  // 16-byte vectors of counts a thread keeps between the scan phases
constexpr int kAggBits = 11;  // the count's per-CTA grouping table: 2^11 entries
constexpr int kAggSlots = 1 << kAggBits;
constexpr uint32_t kAggEmpty = 0xffffffffu;  // never a cell index (cells < 2^32 - 1)
static_assert(kAggSlots % kThreads == 0 && 2 * kAggSlots <= kScanVecs * kThreads * 4,
              "grouping table must fit in s_held");

__device__ __forceinline__ uint32_t load_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 load_policy(const uint4 *p, unsigned long long policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void arrive_release(uint32_t *p) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}

// Thread 0 of every CTA counts the barriers it has passed in `passed`.  The
// __syncthreads before the arrival makes the CTA's writes visible to thread 0,
// whose release add publishes them; the acquire loads that see every arrival
// make the other CTAs' writes visible, and the closing __syncthreads hands
// them to the whole CTA.  A CTA may do work of its own between grid_arrive
// and grid_wait, as long as that work neither writes what other CTAs read
// after the barrier nor reads what they write before it.
__device__ __forceinline__ void grid_arrive(grid_ws_header *hdr, uint32_t &passed) {
    __syncthreads();
    if (threadIdx.x == 0) {
        passed += 1u;
        arrive_release(&hdr->bar_count);
    }
}

__device__ inline void grid_wait(grid_ws_header *hdr, uint32_t passed) {
    if (threadIdx.x == 0) {
        const uint32_t target = passed * gridDim.x + *reinterpret_cast<volatile uint32_t *>(&hdr->bar_extra);
        if (load_acquire(&hdr->bar_count) < target) {
            const unsigned long long start = global_ns();
            uint32_t polls = 0;
            while (load_acquire(&hdr->bar_count) < target) {
                if ((++polls & 31u) == 0 && global_ns() - start > kSpinLimitNs) {
                    record_status(&hdr->status, kStatusTimeout);
                    break;
                }
            }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void grid_barrier(grid_ws_header *hdr, uint32_t &passed) {
    grid_arrive(hdr, passed);
    grid_wait(hdr, passed);
}

// Block-wide sum (every thread gets it).
__device__ inline uint32_t block_sum(uint32_t v, uint32_t *s_red) {
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane_id() == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += s_red[w];
    __syncthreads();
    return t;
}

// Exclusive scans of the first kRows rows at once: row q holds one value per
// thread (t[q]); excl[q] receives the thread's exclusive prefix within row q
// and rows[q] the row's total (zero for the rows past kRows).  Each warp
// scans its lanes with shuffles; warp 0 then scans the warps' totals of every
// row (kWarps lanes per row) and leaves the prefixes in s_rows, row kScanVecs
// holding the rows' totals.  Three __syncthreads for all rows.
static_assert(32 % kWarps == 0 && (kScanVecs * kWarps) % 32 == 0 && kScanVecs <= kWarps,
              "warp 0 scans the warp totals of all rows in segments of kWarps lanes");
template <int kRows = kScanVecs>
__device__ __forceinline__ void rows_exclusive_scan(const uint32_t (&t)[kScanVecs],
                                                    uint32_t (&excl)[kScanVecs],
                                                    uint32_t (&rows)[kScanVecs],
                                                    uint32_t (*s_rows)[kWarps]) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t incl[kScanVecs];
#pragma unroll
    for (int q = 0; q < kRows; ++q) incl[q] = t[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const uint32_t up = __shfl_up_sync(0xffffffffu, incl[q], o);
            if (lane >= (uint32_t)o) incl[q] += up;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int q = 0; q < kRows; ++q) s_rows[q][warp] = incl[q];
    }
    __syncthreads();
    if (warp == 0) {
        // Entry e = j * 32 + lane of the flattened [kScanVecs][kWarps] table.
        constexpr int kPer = (kRows * kWarps + 31) / 32;
        const uint32_t seg = lane % kWarps;
        uint32_t x[kPer], v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) v[j] = x[j] = j * 32 + lane < kRows * kWarps ? (&s_rows[0][0])[j * 32 + lane] : 0u;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const uint32_t up = __shfl_up_sync(0xffffffffu, v[j], o, kWarps);
                if (seg >= (uint32_t)o) v[j] += up;
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (j * 32 + lane < kRows * kWarps) {
                (&s_rows[0][0])[j * 32 + lane] = v[j] - x[j];
                if (seg == kWarps - 1) s_rows[kScanVecs][(j * 32 + lane) / kWarps] = v[j];
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) {
        excl[q] = q < kRows ? s_rows[q][warp] + incl[q] - t[q] : 0u;
        rows[q] = q < kRows ? s_rows[kScanVecs][q] : 0u;
    }
    __syncthreads();
}

// Four counts starting at cell c (a multiple of 4), zeros past `hi`.
__device__ __forceinline__ uint4 load_counts(const uint32_t *conteos, uint64_t c, uint64_t hi) {
    if (c + 4 <= hi) return *reinterpret_cast<const uint4 *>(conteos + c);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c < hi) v.x = conteos[c];
    if (c + 1 < hi) v.y = conteos[c + 1];
    if (c + 2 < hi) v.z = conteos[c + 2];
    return v;
}

// inicios[c..c+3] = first, first + v.x, ... (only cells below `hi`).
__device__ __forceinline__ void store_starts(uint32_t *inicios, uint64_t c, uint64_t hi, uint32_t first,
                                             const uint4 &v) {
    const uint4 o = make_uint4(first, first + v.x, first + v.x + v.y, first + v.x + v.y + v.z);
    if (c + 4 <= hi) {
        *reinterpret_cast<uint4 *>(inicios + c) = o;
    } else {
        if (c < hi) inicios[c] = o.x;
        if (c + 1 < hi) inicios[c + 1] = o.y;
        if (c + 2 < hi) inicios[c + 2] = o.z;
    }
}

// conteos[c..c+3] = v (the histogram) and counts[c..c+3] = 0 (only cells
// below `hi`).
__device__ __forceinline__ void store_counts(uint32_t *conteos, uint32_t *counts, uint64_t c, uint64_t hi,
                                             const uint4 &v) {
    if (c + 4 <= hi) {
        *reinterpret_cast<uint4 *>(conteos + c) = v;
        *reinterpret_cast<uint4 *>(counts + c) = make_uint4(0u, 0u, 0u, 0u);
    } else {
        const uint32_t w[3] = {v.x, v.y, v.z};
        for (int k = 0; k < 3; ++k) {
            if (c + k < hi) {
                conteos[c + k] = w[k];
                counts[c + k] = 0u;
            }
        }
    }
}

// Workspace arrays of the fused build.
struct FusedScratch {
    uint32_t *chunk_sums;      // per-CTA chunk totals
    uint32_t *slots;           // per-particle slot in its cell
    uint32_t *counts;          // per-cell counters, zero between builds
    uint32_t *queue;           // stable mode: cells longer than kRegisterMax
    uint32_t queue_capacity;
    uint32_t *sort_scratch;    // stable mode: radix ping-pong buffer (N words)
};


// Per-launch arguments of a build.
struct BuildArgs {
    const uint4 *origen;
    uint4 *destino;
    uint32_t *conteos;
    uint32_t *celdaDe;
    uint32_t *inicios;
    uint32_t *ordenado;
    uint32_t n;
    uint64_t cells;
};

// This CTA's share of the particles: one contiguous, equal range.
__device__ __forceinline__ void particle_range(uint32_t n, uint64_t &lo, uint64_t &hi) {
    lo = (uint64_t)n * blockIdx.x / gridDim.x;
    hi = (uint64_t)n * (blockIdx.x + 1) / gridDim.x;
}

// Zero the workspace counters (grid-stride).
__device__ __forceinline__ void clear_counters(uint32_t *counts, uint64_t cells) {
    const uint64_t quads = cells / 4;
    const uint64_t grid_threads = (uint64_t)gridDim.x * kThreads;
    uint4 *c4 = reinterpret_cast<uint4 *>(counts);
    for (uint64_t q = (uint64_t)blockIdx.x * kThreads + threadIdx.x; q < quads; q += grid_threads)
        c4[q] = make_uint4(0u, 0u, 0u, 0u);
    for (uint64_t c = quads * 4 + (uint64_t)blockIdx.x * kThreads + threadIdx.x; c < cells; c += grid_threads)
        counts[c] = 0u;
}

// ---- count: cell, histogram and slot ----------------------------------------
// With kFromPositions the cell of particle i is computed from its record and
// saved in celdaDe[i]; otherwise it is read back from celdaDe.  Each round the
// CTA groups its particles by cell in a shared-memory hash table (s_held is
// free until the scan): the particles of a cell that claims an entry take
// their slots with one global atomic for the whole group, so a crowded cell
// costs one atomic per CTA and round rather than one per particle ("Contar
// partículas por celda", §La contención de las celdas densas: aggregate, then
// one contribution per group).  A particle whose entry another cell holds
// takes its slot directly.  The records are read with an L2 evict-last
// policy, so they are still in L2 when they are moved.
template <bool kFromPositions>
__device__ __forceinline__ void count_phase(const BuildArgs &a, const Geometry &g, const FusedScratch &ws,
                                            uint64_t p_lo, uint64_t p_hi, uint4 (*s_held)[kThreads]) {
    const uint32_t tid = threadIdx.x;
    unsigned long long keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    uint32_t *s_key = reinterpret_cast<uint32_t *>(&s_held[0][0]);  // [kAggSlots] cell or kAggEmpty
    uint32_t *s_cnt = s_key + kAggSlots;                              // [kAggSlots] count, then base
    for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kCountItems) {
        uint32_t cell[kCountItems];
        if (kFromPositions) {
            uint4 rec[kCountItems];
#pragma unroll
            for (int k = 0; k < kCountItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) rec[k] = load_policy(a.origen + 2 * i, keep);
            }
#pragma unroll
            for (int k = 0; k < kCountItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) {
                    cell[k] = cell_of(rec[k], g);
                    a.celdaDe[i] = cell[k];
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < kCountItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) cell[k] = a.celdaDe[i];
            }
        }
#pragma unroll
        for (int e = 0; e < kAggSlots / kThreads; ++e) {
            s_key[e * kThreads + tid] = kAggEmpty;
            s_cnt[e * kThreads + tid] = 0u;
        }
        __syncthreads();
        uint32_t entry[kCountItems], rank[kCountItems];
#pragma unroll
        for (int k = 0; k < kCountItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            entry[k] = kAggEmpty;
            if (i < p_hi) {
                const uint32_t c = cell[k];
                const uint32_t h = (c * 0x9E3779B1u) >> (32 - kAggBits);
                const uint32_t held = atomicCAS(&s_key[h], kAggEmpty, c);
                if (held == kAggEmpty || held == c) {
                    entry[k] = h;
                    rank[k] = atomicAdd(&s_cnt[h], 1u);
                } else {
                    rank[k] = atomicAdd(ws.counts + c, 1u);
                }
            }
        }
        __syncthreads();
        // One atomic per claimed entry; the entry's count becomes its base slot.
        uint32_t group[kAggSlots / kThreads];
#pragma unroll
        for (int e = 0; e < kAggSlots / kThreads; ++e) {
            const uint32_t m = s_cnt[e * kThreads + tid];
            group[e] = m ? atomicAdd(ws.counts + s_key[e * kThreads + tid], m) : 0u;
        }
#pragma unroll
        for (int e = 0; e < kAggSlots / kThreads; ++e) s_cnt[e * kThreads + tid] = group[e];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kCountItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) ws.slots[i] = entry[k] == kAggEmpty ? rank[k] : s_cnt[entry[k]] + rank[k];
        }
        __syncthreads();  // the table is cleared at the top of the next round
    }
}

// ---- scan over the counters, in one contiguous chunk of cells per CTA --------
// Chunks are multiples of 4 cells so that 16-byte accesses stay aligned.  When
// a chunk fits in kScanVecs vectors per thread its counts stay in s_held
// between the two halves.
struct ScanChunk {
    uint64_t lo, hi;
    bool resident;
};

__device__ __forceinline__ ScanChunk scan_chunk(uint64_t cells) {
    const uint64_t chunk = ((cells + gridDim.x - 1) / gridDim.x + 3) & ~3ull;
    ScanChunk k;
    k.lo = min((uint64_t)blockIdx.x * chunk, cells);
    k.hi = min(k.lo + chunk, cells);
    k.resident = chunk <= 4ull * kThreads * kScanVecs;
    return k;
}

// Scan, first half: this chunk's total in chunk_sums[blockIdx.x].
__device__ __forceinline__ void scan_totals_phase(const FusedScratch &ws, const ScanChunk &k,
                                                  uint4 (*s_held)[kThreads], uint32_t *s_red) {
    const uint32_t tid = threadIdx.x;
    uint32_t sum = 0;
    if (k.resident) {
        uint4 v[kScanVecs];
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) v[q] = load_counts(ws.counts, k.lo + 4ull * (q * kThreads + tid), k.hi);
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) {
            s_held[q][tid] = v[q];
            sum += v[q].x + v[q].y + v[q].z + v[q].w;
        }
    } else {
        for (uint64_t c0 = k.lo; c0 < k.hi; c0 += 4ull * kThreads * kScanVecs) {
            uint4 v[kScanVecs];
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) v[q] = load_counts(ws.counts, c0 + 4ull * (q * kThreads + tid), k.hi);
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) sum += v[q].x + v[q].y + v[q].z + v[q].w;
        }
    }
    sum = block_sum(sum, s_red);
    if (tid == 0) ws.chunk_sums[blockIdx.x] = sum;
}

// Scan, second half: inicios over the chunk, conteos = the counts, the
// counters back to zero; the last CTA writes inicios[C] = N.
__device__ __forceinline__ void scan_starts_phase(const BuildArgs &a, const FusedScratch &ws, const ScanChunk &k,
                                                  uint4 (*s_held)[kThreads], uint32_t *s_red,
                                                  uint32_t (*s_rows)[kWarps]) {
    const uint32_t tid = threadIdx.x;
    uint32_t before = 0;
    for (uint32_t b = tid; b < blockIdx.x; b += kThreads) before += ws.chunk_sums[b];
    uint32_t prefix = block_sum(before, s_red);
    for (uint64_t c0 = k.lo; c0 < k.hi; c0 += 4ull * kThreads * kScanVecs) {
        uint4 v[kScanVecs];
        uint32_t t[kScanVecs];
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) {
            v[q] = k.resident ? s_held[q][tid] : load_counts(ws.counts, c0 + 4ull * (q * kThreads + tid), k.hi);
            t[q] = v[q].x + v[q].y + v[q].z + v[q].w;
        }
        // All kScanVecs rows at once: warp scans, then one exchange of the
        // warp totals through shared memory.
        uint32_t excl[kScanVecs], rows[kScanVecs];
        rows_exclusive_scan(t, excl, rows, s_rows);
        uint32_t row_base = prefix;
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) {
            const uint64_t c = c0 + 4ull * (q * kThreads + tid);
            store_starts(a.inicios, c, k.hi, row_base + excl[q], v[q]);
            store_counts(a.conteos, ws.counts, c, k.hi, v[q]);
            row_base += rows[q];
        }
        prefix = row_base;
    }
    if (blockIdx.x == gridDim.x - 1 && tid == 0) a.inicios[a.cells] = prefix;
}

// ---- scatter with the records: ordenado and destino in one pass --------------
// Particle i's place k = inicios[c] + slots[i] is known here, so its record
// goes straight to destino[k] ("Reordenar por celda…", §El kernel de
// reordenación, applied from the source side: the same permutation as the
// gather destino[k] = origen[ordenado[k]]).  Two threads carry one record (a
// 16-byte half each), so every pair writes one whole 32-byte sector; the reads
// of origen are coalesced and hit the sectors the count kept in L2.
__device__ __forceinline__ void scatter_move_phase(const BuildArgs &a, const FusedScratch &ws, uint32_t *status,
                                                   uint64_t p_lo, uint64_t p_hi) {
    const uint32_t tid = threadIdx.x;
    unsigned long long last_use;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(last_use));
    const uint64_t h_lo = 2 * p_lo, h_hi = 2 * p_hi;
    for (uint64_t r0 = h_lo; r0 < h_hi; r0 += (uint64_t)kThreads * kMoveItems) {
        uint32_t cell[kMoveItems], slot[kMoveItems], start[kMoveItems];
        uint4 v[kMoveItems];
#pragma unroll
        for (int k = 0; k < kMoveItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            if (h < h_hi) {
                cell[k] = a.celdaDe[h >> 1];
                slot[k] = ws.slots[h >> 1];
                v[k] = load_policy(a.origen + h, last_use);
            }
        }
#pragma unroll
        for (int k = 0; k < kMoveItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            if (h < h_hi) start[k] = a.inicios[cell[k]];
        }
#pragma unroll
        for (int k = 0; k < kMoveItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            if (h < h_hi) {
                const uint32_t pos = start[k] + slot[k];
                if (pos < a.n) {
                    store_cs(a.destino + 2 * (uint64_t)pos + (h & 1), v[k]);
                    if ((h & 1) == 0) a.ordenado[pos] = (uint32_t)(h >> 1);
                } else if ((h & 1) == 0) {
                    record_status(status, kStatusBounds);
                }
            }
        }
    }
}

// ---- stable tail: scatter the indices, sort each cell, then gather -------------
// ("Construir el índice…", §El orden dentro de la celda: particle index as the
// tie-break.)  The scatter places particle i at inicios[c] + slots[i]; one
// thread per cell sorts its segment in registers when it holds at most 32
// particles and queues it otherwise; CTAs then take the queued segments one
// each (bitonic in shared memory up to 8192, an LSD radix sort through the
// workspace beyond); finally the records are gathered in the sorted order.
__device__ __forceinline__ void stable_tail_phase(const BuildArgs &a, const FusedScratch &ws, grid_ws_header *hdr,
                                                  uint32_t &passed, uint64_t p_lo, uint64_t p_hi,
                                                  uint4 (*s_held)[kThreads]) {
    const uint32_t tid = threadIdx.x;
    const uint32_t ctas = gridDim.x;
    for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kScatterItems) {
        uint32_t cell[kScatterItems], slot[kScatterItems], start[kScatterItems];
#pragma unroll
        for (int k = 0; k < kScatterItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) {
                cell[k] = a.celdaDe[i];
                slot[k] = ws.slots[i];
            }
        }
#pragma unroll
        for (int k = 0; k < kScatterItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) start[k] = a.inicios[cell[k]];
        }
#pragma unroll
        for (int k = 0; k < kScatterItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) {
                const uint32_t pos = start[k] + slot[k];
                if (pos < a.n)
                    a.ordenado[pos] = (uint32_t)i;
                else
                    record_status(&hdr->status, kStatusBounds);
            }
        }
    }
    grid_barrier(hdr, passed);

    // Every cell's segment sorted by particle index ("Construir el
    // índice…", §El orden dentro de la celda).  Short segments are sorted
    // by one thread in registers; longer ones are queued.
    const uint64_t grid_threads = (uint64_t)ctas * kThreads;
    for (uint64_t c = (uint64_t)blockIdx.x * kThreads + tid; c < a.cells; c += grid_threads) {
        const uint32_t s = a.inicios[c];
        if (!sort_short_segment(a.ordenado + s, a.inicios[c + 1] - s)) {
            const uint32_t q = atomicAdd(&hdr->stable_big, 1u);
            if (q < ws.queue_capacity)
                ws.queue[q] = (uint32_t)c;
            else
                record_status(&hdr->status, kStatusBounds);
        }
    }
    grid_barrier(hdr, passed);
    // Long segments, one CTA each: bitonic in shared memory up to 8192
    // indices, radix through the workspace scratch beyond.
    const uint32_t queued = *reinterpret_cast<volatile uint32_t *>(&hdr->stable_big);
    const uint32_t count = min(queued, ws.queue_capacity);
    uint32_t *s_buf = reinterpret_cast<uint32_t *>(&s_held[0][0]);
    for (uint32_t q = blockIdx.x; q < count; q += ctas) {
        const uint32_t c = ws.queue[q];
        const uint32_t s = a.inicios[c];
        sort_long_segment<kThreads>(a.ordenado + s, ws.sort_scratch + s, a.inicios[c + 1] - s, a.n, s_buf,
                                    kScanVecs * kThreads * 4);
    }
    grid_barrier(hdr, passed);

    // Gather, two threads per 32-byte record.
    unsigned long long last_use;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(last_use));
    const uint64_t h_lo = 2 * p_lo, h_hi = 2 * p_hi;
    for (uint64_t r0 = h_lo; r0 < h_hi; r0 += (uint64_t)kThreads * kGatherItems) {
        uint32_t src[kGatherItems];
#pragma unroll
        for (int k = 0; k < kGatherItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            src[k] = h < h_hi ? a.ordenado[h >> 1] : 0u;
        }
        uint4 v[kGatherItems];
#pragma unroll
        for (int k = 0; k < kGatherItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            if (h < h_hi && src[k] < a.n) v[k] = load_policy(a.origen + 2 * (uint64_t)src[k] + (h & 1), last_use);
        }
#pragma unroll
        for (int k = 0; k < kGatherItems; ++k) {
            const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
            if (h < h_hi) {
                if (src[k] < a.n)
                    store_cs(a.destino + h, v[k]);
                else if ((h & 1) == 0)
                    record_status(&hdr->status, kStatusBounds);
            }
        }
    }
}

// The last CTA out of a launch resets the barrier counter for the next one.
__device__ __forceinline__ void leave_launch(grid_ws_header *hdr) {
    if (threadIdx.x == 0 && atomicAdd(&hdr->bar_exit, 1u) == gridDim.x - 1u) {
        hdr->bar_count = 0u;
        hdr->bar_exit = 0u;
    }
}

}  // namespace fused
}  // namespace ugrid
