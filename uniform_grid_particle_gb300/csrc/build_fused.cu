// The whole grid build in one cooperative launch.
//
// The pages chain separate dispatches because the phases depend on each other
// across workgroups ("Construir el índice de la rejilla…", §La cadena
// completa: the scan needs every count, the scatter every start).  Here every
// CTA of the grid is resident at once (cooperative launch, two CTAs per SM),
// so a grid-wide barrier stands in for each kernel boundary:
//
//   count   celdaDe[i] = cell of particle i; the atomic that counts it in the
//           workspace counter array returns its slot in the cell, kept in
//           slots[i]  ("Contar partículas por celda", §El kernel; the counter
//           array is also the cursor of "La dispersión").  Particles of one
//           CTA that share a cell are grouped first and take their slots with
//           one atomic (§La contención de las celdas densas)
//   scan a  each CTA totals one contiguous chunk of the counters
//   scan b  each CTA adds the totals of the chunks before it, scans its chunk
//           into inicios, copies the counts to conteos and zeroes its
//           counters; the last CTA writes inicios[C] = N
//                                                     ("Del conteo al inicio")
//   scatter ordenado[inicios[c] + slots[i]] = i        ("La dispersión")
//           and, in the same pass, destino[inicios[c] + slots[i]] = origen[i]
//
// The last line is the pages' gather destino[k] = origen[ordenado[k]] ("El
// kernel de reordenación") applied from the other side: the same permutation
// gives the same destino, and the phase, its barrier and the re-read of
// ordenado disappear.  Stable mode keeps a separate gather, because its
// places are known only once every cell's segment is sorted.
//
// Because the count's atomic already hands out the slot, the pages' second
// clear and second atomic pass are not needed: conteos ends as the histogram,
// exactly as after their cursor scatter, and every output is one the pages'
// chain can produce (order inside a cell is the atomics' arrival order).
//
// The counters live in the workspace and every build leaves them zero (scan b
// zeroes them after reading), so no clear phase is needed ("Poner a cero" is
// done by the previous build).  A header word records that they are clean; it
// is dropped while a build is using them, so a build that did not finish
// makes the next one clear them first.
//
// With GRID_STABLE two phases follow the scatter: one thread per cell sorts
// its segment in registers when it holds at most 32 particles and queues it
// otherwise, then CTAs take the queued segments one each (bitonic in shared
// memory up to 8192, an LSD radix sort through the workspace beyond).
//
// Particles (and the gather's half-records) are split into one contiguous,
// equal range per CTA, so every CTA has the same work in every phase.
//
// The count reads each record's first 16 bytes with an L2 evict-last policy
// and the record move (or the stable gather) reads the records with
// evict-first: the 32-byte sectors the count brings into L2 are still there
// when the records move.
//
// Grid barriers: a CTA arrives with a release add on a counter that only grows
// during the launch and waits, with acquire loads, until it reaches the number
// of CTAs times the barriers passed; the last CTA to leave the kernel resets
// it.  A wait gives up after kSpinLimitNs and records kStatusTimeout, so the
// kernel cannot hang (co-residency is guaranteed by the cooperative launch, so
// the limit is a guard, not part of the protocol).
#include <atomic>

#include "segsort_device.cuh"

namespace ugrid {
namespace {

// Measurement hook at each phase boundary; compiled out unless a profiling
// build defines it.
#ifndef UGRID_PHASE_MARK
#define UGRID_PHASE_MARK(phase)
#endif
#ifndef UGRID_PHASE_END
#define UGRID_PHASE_END(phase)
#endif

#ifndef UGRID_FUSED_COUNT_ITEMS
#define UGRID_FUSED_COUNT_ITEMS 4
#endif
#ifndef UGRID_FUSED_SCATTER_ITEMS
#define UGRID_FUSED_SCATTER_ITEMS 8
#endif
#ifndef UGRID_FUSED_GATHER_ITEMS
#define UGRID_FUSED_GATHER_ITEMS 4
#endif
#ifndef UGRID_FUSED_MOVE_ITEMS
#define UGRID_FUSED_MOVE_ITEMS 4
#endif

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCountItems = UGRID_FUSED_COUNT_ITEMS;      // particles per thread per round
constexpr int kScatterItems = UGRID_FUSED_SCATTER_ITEMS;  // particles per thread per round
constexpr int kGatherItems = UGRID_FUSED_GATHER_ITEMS;    // half-records per thread per round
constexpr int kMoveItems = UGRID_FUSED_MOVE_ITEMS;        // half-records per thread per round
constexpr int kScanVecs = 4;  // 16-byte vectors of counts a thread keeps between the scan phases
constexpr int kAggBits = 11;  // the count's per-CTA grouping table: 2^11 entries
constexpr int kAggSlots = 1 << kAggBits;
constexpr uint32_t kAggEmpty = 0xffffffffu;  // never a cell index (cells < 2^32 - 1)
static_assert(kAggSlots % kThreads == 0 && 2 * kAggSlots <= kScanVecs * kThreads * 4,
              "grouping table must fit in s_held");
constexpr int kMaxDevices = 64;

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
// them to the whole CTA.
__device__ void grid_barrier(grid_ws_header *hdr, uint32_t &passed) {
    __syncthreads();
    if (threadIdx.x == 0) {
        passed += 1u;
        const uint32_t target = passed * gridDim.x;
        arrive_release(&hdr->bar_count);
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

// Block-wide sum (every thread gets it).
__device__ uint32_t block_sum(uint32_t v, uint32_t *s_red) {
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane_id() == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += s_red[w];
    __syncthreads();
    return t;
}

// Exclusive scans of kScanVecs rows at once: row q holds one value per
// thread (t[q]); excl[q] receives the thread's exclusive prefix within row q
// and rows[q] the row's total.  Two __syncthreads for all rows.
__device__ __forceinline__ void rows_exclusive_scan(const uint32_t (&t)[kScanVecs],
                                                    uint32_t (&excl)[kScanVecs],
                                                    uint32_t (&rows)[kScanVecs],
                                                    uint32_t (*s_rows)[kWarps]) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t incl[kScanVecs];
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) incl[q] = t[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) {
            const uint32_t up = __shfl_up_sync(0xffffffffu, incl[q], o);
            if (lane >= (uint32_t)o) incl[q] += up;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) s_rows[q][warp] = incl[q];
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) {
        uint32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t x = s_rows[q][w];
            before += (uint32_t)w < warp ? x : 0u;
            total += x;
        }
        excl[q] = before + incl[q] - t[q];
        rows[q] = total;
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

template <bool kStable>
__global__ void __launch_bounds__(kThreads, 2)
build_fused_kernel(const uint4 *__restrict__ origen, uint4 *__restrict__ destino,
                   uint32_t *__restrict__ conteos, uint32_t *__restrict__ celdaDe,
                   uint32_t *__restrict__ inicios, uint32_t *__restrict__ ordenado, uint32_t n,
                   uint64_t cells, Geometry g, grid_ws_header *hdr, FusedScratch ws) {
    uint32_t *__restrict__ chunk_sums = ws.chunk_sums;
    uint32_t *__restrict__ slots = ws.slots;
    uint32_t *__restrict__ counts = ws.counts;
    __shared__ uint32_t s_red[kWarps];
    __shared__ uint4 s_held[kScanVecs][kThreads];  // this CTA's chunk of counts (32 KB)
    __shared__ uint32_t s_clean;
    __shared__ uint32_t s_rows[kScanVecs][kWarps];
    const uint32_t tid = threadIdx.x;
    const uint32_t ctas = gridDim.x;
    uint32_t passed = 0;  // grid barriers passed (thread 0)
    // Read before this CTA's first arrival, hence before anyone changes it.
    if (tid == 0) s_clean = *reinterpret_cast<volatile uint32_t *>(&hdr->counts_clean) >= cells;
    // Nobody touches the long-segment queue before the stable phases.
    if (kStable && blockIdx.x == 0 && tid == 0) hdr->stable_big = 0u;
    __syncthreads();
    // This CTA's particles: one contiguous, equal share.
    const uint64_t p_lo = (uint64_t)n * blockIdx.x / ctas;
    const uint64_t p_hi = (uint64_t)n * (blockIdx.x + 1) / ctas;

    UGRID_PHASE_MARK(0);
    // ---- clear the counters, only if the previous build did not leave them zero
    if (!s_clean) {
        const uint64_t quads = cells / 4;
        const uint64_t grid_threads = (uint64_t)ctas * kThreads;
        uint4 *c4 = reinterpret_cast<uint4 *>(counts);
        for (uint64_t q = (uint64_t)blockIdx.x * kThreads + tid; q < quads; q += grid_threads)
            c4[q] = make_uint4(0u, 0u, 0u, 0u);
        for (uint64_t c = quads * 4 + (uint64_t)blockIdx.x * kThreads + tid; c < cells; c += grid_threads)
            counts[c] = 0u;
        grid_barrier(hdr, passed);
    }

    UGRID_PHASE_MARK(1);
    // ---- count: cell, histogram and slot -------------------------------------
    unsigned long long keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    // Each round the CTA groups its particles by cell in a shared-memory hash
    // table (the counts' s_held space is free until scan a): the particles of a
    // cell that claims an entry take their slots with one global atomic for the
    // whole group, so a crowded cell costs one atomic per CTA and round rather
    // than one per particle ("Contar partículas por celda", §La contención de
    // las celdas densas: aggregate, then one contribution per group).  A
    // particle whose entry another cell holds takes its slot directly.
    uint32_t *s_key = reinterpret_cast<uint32_t *>(&s_held[0][0]);  // [kAggSlots] cell or kAggEmpty
    uint32_t *s_cnt = s_key + kAggSlots;                              // [kAggSlots] count, then base
    for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kCountItems) {
        uint4 rec[kCountItems];
#pragma unroll
        for (int k = 0; k < kCountItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) rec[k] = load_policy(origen + 2 * i, keep);
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
                const uint32_t c = cell_of(rec[k], g);
                celdaDe[i] = c;
                const uint32_t h = (c * 0x9E3779B1u) >> (32 - kAggBits);
                const uint32_t held = atomicCAS(&s_key[h], kAggEmpty, c);
                if (held == kAggEmpty || held == c) {
                    entry[k] = h;
                    rank[k] = atomicAdd(&s_cnt[h], 1u);
                } else {
                    rank[k] = atomicAdd(counts + c, 1u);
                }
            }
        }
        __syncthreads();
        // One atomic per claimed entry; the entry's count becomes its base slot.
        uint32_t group[kAggSlots / kThreads];
#pragma unroll
        for (int e = 0; e < kAggSlots / kThreads; ++e) {
            const uint32_t m = s_cnt[e * kThreads + tid];
            group[e] = m ? atomicAdd(counts + s_key[e * kThreads + tid], m) : 0u;
        }
#pragma unroll
        for (int e = 0; e < kAggSlots / kThreads; ++e) s_cnt[e * kThreads + tid] = group[e];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kCountItems; ++k) {
            const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
            if (i < p_hi) slots[i] = entry[k] == kAggEmpty ? rank[k] : s_cnt[entry[k]] + rank[k];
        }
        __syncthreads();  // the table is cleared at the top of the next round
    }
    UGRID_PHASE_END(1);
    grid_barrier(hdr, passed);
    // The counters are not zero until scan b has run to the end.
    if (blockIdx.x == 0 && tid == 0) hdr->counts_clean = 0u;

    UGRID_PHASE_MARK(2);
    // ---- scan a: chunk totals --------------------------------------------------
    // Chunks are multiples of 4 cells so that 16-byte accesses stay aligned.
    // When a chunk fits in kScanVecs vectors per thread its counts stay in
    // shared memory for scan b; otherwise scan b reads them again.
    const uint64_t chunk = ((cells + ctas - 1) / ctas + 3) & ~3ull;
    const uint64_t lo = min((uint64_t)blockIdx.x * chunk, cells);
    const uint64_t hi = min(lo + chunk, cells);
    const bool resident = chunk <= 4ull * kThreads * kScanVecs;
    {
        uint32_t sum = 0;
        if (resident) {
            uint4 v[kScanVecs];
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) v[q] = load_counts(counts, lo + 4ull * (q * kThreads + tid), hi);
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) {
                s_held[q][tid] = v[q];
                sum += v[q].x + v[q].y + v[q].z + v[q].w;
            }
        } else {
            for (uint64_t c0 = lo; c0 < hi; c0 += 4ull * kThreads * kScanVecs) {
                uint4 v[kScanVecs];
#pragma unroll
                for (int q = 0; q < kScanVecs; ++q) v[q] = load_counts(counts, c0 + 4ull * (q * kThreads + tid), hi);
#pragma unroll
                for (int q = 0; q < kScanVecs; ++q) sum += v[q].x + v[q].y + v[q].z + v[q].w;
            }
        }
        sum = block_sum(sum, s_red);
        if (tid == 0) chunk_sums[blockIdx.x] = sum;
    }
    UGRID_PHASE_END(2);
    grid_barrier(hdr, passed);

    UGRID_PHASE_MARK(3);
    // ---- scan b: starts, histogram copy, counters back to zero ---------------
    {
        uint32_t before = 0;
        for (uint32_t b = tid; b < blockIdx.x; b += kThreads) before += chunk_sums[b];
        uint32_t prefix = block_sum(before, s_red);
        for (uint64_t c0 = lo; c0 < hi; c0 += 4ull * kThreads * kScanVecs) {
            uint4 v[kScanVecs];
            uint32_t t[kScanVecs];
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) {
                v[q] = resident ? s_held[q][tid] : load_counts(counts, c0 + 4ull * (q * kThreads + tid), hi);
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
                store_starts(inicios, c, hi, row_base + excl[q], v[q]);
                store_counts(conteos, counts, c, hi, v[q]);
                row_base += rows[q];
            }
            prefix = row_base;
        }
        if (blockIdx.x == ctas - 1 && tid == 0) inicios[cells] = prefix;
    }
    UGRID_PHASE_END(3);
    grid_barrier(hdr, passed);
    // Every CTA zeroed its counters before that barrier.
    if (blockIdx.x == 0 && tid == 0 && (hdr->status & kStatusTimeout) == 0)
        hdr->counts_clean = (uint32_t)cells;

    UGRID_PHASE_MARK(4);
    if constexpr (!kStable) {
        // ---- scatter with the records: ordenado and destino in one pass -----
        // Particle i's place k = inicios[c] + slots[i] is known here, so its
        // record goes straight to destino[k] instead of being fetched back
        // through ordenado[k] after another grid barrier.  Two threads carry
        // one record (a 16-byte half each), so every pair writes one whole
        // 32-byte sector; the reads of origen are coalesced and hit the
        // sectors the count kept in L2.
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
                    cell[k] = celdaDe[h >> 1];
                    slot[k] = slots[h >> 1];
                    v[k] = load_policy(origen + h, last_use);
                }
            }
#pragma unroll
            for (int k = 0; k < kMoveItems; ++k) {
                const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
                if (h < h_hi) start[k] = inicios[cell[k]];
            }
#pragma unroll
            for (int k = 0; k < kMoveItems; ++k) {
                const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
                if (h < h_hi) {
                    const uint32_t pos = start[k] + slot[k];
                    if (pos < n) {
                        store_cs(destino + 2 * (uint64_t)pos + (h & 1), v[k]);
                        if ((h & 1) == 0) ordenado[pos] = (uint32_t)(h >> 1);
                    } else if ((h & 1) == 0) {
                        record_status(&hdr->status, kStatusBounds);
                    }
                }
            }
        }
    } else {
        // ---- stable mode: scatter the indices, sort each cell, then gather -------
        for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kScatterItems) {
            uint32_t cell[kScatterItems], slot[kScatterItems], start[kScatterItems];
#pragma unroll
            for (int k = 0; k < kScatterItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) {
                    cell[k] = celdaDe[i];
                    slot[k] = slots[i];
                }
            }
#pragma unroll
            for (int k = 0; k < kScatterItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) start[k] = inicios[cell[k]];
            }
#pragma unroll
            for (int k = 0; k < kScatterItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) {
                    const uint32_t pos = start[k] + slot[k];
                    if (pos < n)
                        ordenado[pos] = (uint32_t)i;
                    else
                        record_status(&hdr->status, kStatusBounds);
                }
            }
        }
        UGRID_PHASE_END(4);
        grid_barrier(hdr, passed);

        {
            // ---- every cell's segment sorted by particle index -------------------
            // ("Construir el índice…", §El orden dentro de la celda.)  Short
            // segments are sorted by one thread in registers; longer ones are queued.
            const uint64_t grid_threads = (uint64_t)ctas * kThreads;
            for (uint64_t c = (uint64_t)blockIdx.x * kThreads + tid; c < cells; c += grid_threads) {
                const uint32_t a = inicios[c];
                if (!sort_short_segment(ordenado + a, inicios[c + 1] - a)) {
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
                const uint32_t a = inicios[c];
                sort_long_segment<kThreads>(ordenado + a, ws.sort_scratch + a, inicios[c + 1] - a, n, s_buf,
                                            kScanVecs * kThreads * 4);
            }
            grid_barrier(hdr, passed);
        }

        UGRID_PHASE_MARK(5);
        // ---- gather: two threads per 32-byte record -------------------------------
        unsigned long long last_use;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(last_use));
        const uint64_t h_lo = 2 * p_lo, h_hi = 2 * p_hi;
        for (uint64_t r0 = h_lo; r0 < h_hi; r0 += (uint64_t)kThreads * kGatherItems) {
            uint32_t src[kGatherItems];
#pragma unroll
            for (int k = 0; k < kGatherItems; ++k) {
                const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
                src[k] = h < h_hi ? ordenado[h >> 1] : 0u;
            }
            uint4 v[kGatherItems];
#pragma unroll
            for (int k = 0; k < kGatherItems; ++k) {
                const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
                if (h < h_hi && src[k] < n) v[k] = load_policy(origen + 2 * (uint64_t)src[k] + (h & 1), last_use);
            }
#pragma unroll
            for (int k = 0; k < kGatherItems; ++k) {
                const uint64_t h = r0 + (uint64_t)k * kThreads + tid;
                if (h < h_hi) {
                    if (src[k] < n)
                        store_cs(destino + h, v[k]);
                    else if ((h & 1) == 0)
                        record_status(&hdr->status, kStatusBounds);
                }
            }
        }
    }
    UGRID_PHASE_MARK(6);

    // The last CTA out resets the barrier counter for the next launch.
    if (tid == 0 && atomicAdd(&hdr->bar_exit, 1u) == ctas - 1u) {
        hdr->bar_count = 0u;
        hdr->bar_exit = 0u;
    }
}

std::atomic<int> g_grid[kMaxDevices];  // cached grid size per device (0 = not yet known)

cudaError_t fused_grid(int device, int *grid) {
    if (device >= 0 && device < kMaxDevices) {
        const int cached = g_grid[device].load(std::memory_order_relaxed);
        if (cached != 0) {
            *grid = cached;
            return cached > 0 ? cudaSuccess : cudaErrorNotSupported;
        }
    }
    int coop = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_fused_kernel<true>, kThreads, 0);
    if (e != cudaSuccess) return e;
    int g = coop ? per_sm * sms : -1;
    if (g == 0) g = -1;
    if (g > (int)kFusedMaxCtas) g = (int)kFusedMaxCtas;
    if (device >= 0 && device < kMaxDevices) g_grid[device].store(g, std::memory_order_relaxed);
    *grid = g;
    return g > 0 ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_build_fused(const ugrid_particula *origen, ugrid_particula *destino,
                               uint32_t *conteos, uint32_t *celdaDe, uint32_t *inicios,
                               uint32_t *ordenado, uint32_t n, uint64_t cells, const Geometry &g,
                               grid_ws_header *hdr, uint32_t *chunk_sums, uint32_t *slots,
                               uint32_t *counts, bool stable, uint32_t *queue,
                               uint32_t queue_capacity, uint32_t *sort_scratch, cudaStream_t s) {
    int device = 0, grid = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = fused_grid(device, &grid);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const FusedScratch ws{chunk_sums, slots, counts, queue, queue_capacity, sort_scratch};
    return cudaLaunchKernelEx(&cfg, stable ? build_fused_kernel<true> : build_fused_kernel<false>,
                              reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino),
                              conteos, celdaDe, inicios, ordenado, n, cells, g, hdr, ws);
}

}  // namespace ugrid
