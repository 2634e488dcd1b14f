// The grid build for sparse grids (far more cells than particles), in one
// cooperative launch with a single grid barrier.
//
// The pages' chain ("Construir el índice de la rejilla con un prefix sum",
// §La cadena completa) costs, at a few particles per hundred cells, mostly
// the pass over the cells: the scan of conteos and the writes of conteos and
// inicios (§Del conteo al inicio: the scan costs in proportion to the cells).
// Here every CTA owns one bucket of consecutive cells and one contiguous
// range of particles, and the particles cross from the second to the first
// through one exchange:
//
//   phase 1 (own particles)  celdaDe[i] = cell of particle i ("Contar
//       partículas por celda", §El kernel); the CTA's particles put in bucket
//       order in shared memory and written out as (cell, particle) pairs in
//       its own range of the workspace; for every bucket b, the number of
//       its particles in buckets below b, written to row b of a table.
//   grid barrier
//   phase 2 (own bucket)  the bucket's run of pairs from every CTA (the table
//       gives where each run starts, and the column's sum is the number of
//       particles in lower buckets: the bucket's first position); the counts
//       of its cells, their exclusive scan, conteos and inicios for the whole
//       bucket; the particles placed at inicios[c] + slot (§La dispersión),
//       in stable mode every cell's segment sorted by particle index (§El
//       orden dentro de la celda); ordenado, and destino[k] =
//       origen[ordenado[k]] ("Reordenar por celda…", §El kernel de
//       reordenación).
//
// No global atomics and no counters that must be zero between builds: the
// table is written whole before it is read.  A bucket of more than kHeld
// particles streams its pairs from the workspace instead of holding them.
#include <atomic>

#include "ugrid_internal.cuh"
#include "fused_common.cuh"

namespace ugrid {
namespace {

using fused::kThreads;
using fused::kWarps;
using fused::kScanVecs;

constexpr uint32_t kWindow = kScanVecs * 4u * kThreads;  // cells of one pass of the shared table: 8192
constexpr uint32_t kRowCells = 4u * kThreads;            // cells of one scan row
constexpr uint32_t kHeld = 4096;                         // pairs a CTA holds in shared memory
constexpr uint32_t kRoundItems = 4;                      // records per thread in flight in phase 1
constexpr uint32_t kLongMax = kThreads;                  // long segments queued per round of cells
constexpr size_t kDynamicSmem = (size_t)kWindow * 4 + (size_t)kHeld * 8 + (size_t)kHeld * 4 * 2;
constexpr int kMaxDevices = 64;
static_assert(kSparseMaxParticlesPerCta <= kHeld, "a CTA's particles fit its pair buffer");

struct SparseArgs {
    const uint4 *origen;
    uint4 *destino;
    uint32_t *conteos;
    uint32_t *celdaDe;
    uint32_t *inicios;
    uint32_t *ordenado;
    uint2 *pairs;       // u32x2[n]: (cell, particle), each CTA's range in bucket order
    uint32_t *table;    // u32[(buckets + 1) * gridDim.x]: row b, column s
    uint32_t *scratch;  // stable mode: radix ping-pong buffer (n words)
    uint32_t n;
    uint64_t cells;
    uint32_t width;     // cells per bucket, a multiple of 4
    uint32_t buckets;   // ceil(cells / width) <= gridDim.x < kThreads
    unsigned long long magic;  // ceil(2^64 / width)
};

// Exclusive scan of one value per thread; *total receives the sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *s_red, uint32_t *total) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (uint32_t)o) incl += up;
    }
    if (lane == 31) s_red[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = s_red[w];
        before += (uint32_t)w < warp ? t : 0u;
        all += t;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

// Both sums at once: *sum_a = the CTA's sum of a; *excl_b = this thread's
// exclusive prefix of b, *sum_b = the CTA's sum of b.
__device__ __forceinline__ void pair_scan(uint32_t a, uint32_t b, uint2 *s_red2, uint32_t *sum_a, uint32_t *excl_b,
                                          uint32_t *sum_b) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t incl = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (uint32_t)o) incl += up;
    }
    const uint32_t wa = __reduce_add_sync(0xffffffffu, a);
    if (lane == 31) s_red2[warp] = make_uint2(wa, incl);
    __syncthreads();
    uint32_t before = 0, all_a = 0, all_b = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint2 t = s_red2[w];
        before += (uint32_t)w < warp ? t.y : 0u;
        all_a += t.x;
        all_b += t.y;
    }
    *sum_a = all_a;
    *excl_b = before + incl - b;
    *sum_b = all_b;
}

// The source CTA whose run holds position k of the bucket: the last s with
// off[s] <= k (runs of zero length share their start with the next run).
__device__ __forceinline__ uint32_t source_of(const uint32_t *s_off, uint32_t sources, uint32_t k) {
    uint32_t lo = 0, hi = sources;  // off[lo] <= k < off[hi] (off[sources] = total)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (s_off[mid] <= k)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// The grid barrier's wait (thread 0 polls, bounded); true for every thread
// of the CTA when all CTAs arrived, false after the wait gave up (the
// timeout is recorded in the status word).
__device__ __forceinline__ bool wait_all(grid_ws_header *hdr, uint32_t passed, uint32_t *s_flag) {
    if (threadIdx.x == 0) {
        const uint32_t target = passed * gridDim.x + *reinterpret_cast<volatile uint32_t *>(&hdr->bar_extra);
        uint32_t ok = 1u;
        if (fused::load_acquire(&hdr->bar_count) < target) {
            const unsigned long long start = global_ns();
            uint32_t polls = 0;
            while (fused::load_acquire(&hdr->bar_count) < target) {
                if ((++polls & 31u) == 0 && global_ns() - start > kSpinLimitNs) {
                    record_status(&hdr->status, kStatusTimeout);
                    ok = 0u;
                    break;
                }
            }
        }
        *s_flag = ok;
    }
    __syncthreads();
    const bool ok = *s_flag != 0u;
    __syncthreads();
    return ok;
}

// conteos[c..c+3] = v, only cells below `hi`.
__device__ __forceinline__ void store_four(uint32_t *conteos, uint64_t c, uint64_t hi, const uint4 &v) {
    if (c + 4 <= hi) {
        *reinterpret_cast<uint4 *>(conteos + c) = v;
    } else {
        if (c < hi) conteos[c] = v.x;
        if (c + 1 < hi) conteos[c + 1] = v.y;
        if (c + 2 < hi) conteos[c + 2] = v.z;
    }
}

// One window of the bucket's cells [w0, w0 + kWindow): s_table holds their
// counts.  Writes conteos (only the vectors of four that are not all zero:
// the bucket's conteos were zeroed while the grid barrier filled) and inicios
// (inicios = base + the bucket-local start), and leaves the bucket-local
// starts in s_table; returns the window's particles.  `run` is the
// bucket-local position of the window's first one.
__device__ __forceinline__ uint32_t scan_window(uint32_t *conteos, uint32_t *inicios, uint32_t *s_table, uint64_t w0,
                                                uint64_t hi, uint32_t run, uint32_t base,
                                                uint32_t (*s_rows)[kWarps]) {
    const uint32_t tid = threadIdx.x;
    uint4 *s_vec = reinterpret_cast<uint4 *>(s_table);
    uint32_t t[kScanVecs], excl[kScanVecs], rows[kScanVecs];
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) {
        const uint4 v = s_vec[q * kThreads + tid];
        t[q] = v.x + v.y + v.z + v.w;
    }
    fused::rows_exclusive_scan(t, excl, rows, s_rows);
    uint32_t row_base = run;
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) {
        // Each thread reads back only its own vectors, so they still hold counts.
        const uint4 v = s_vec[q * kThreads + tid];
        const uint32_t first = row_base + excl[q];
        const uint64_t c = w0 + (uint64_t)q * kRowCells + 4u * tid;
        if (v.x | v.y | v.z | v.w) store_four(conteos, c, hi, v);  // zeros written before the barrier
        fused::store_starts(inicios, c, hi, base + first, v);
        s_vec[q * kThreads + tid] = make_uint4(first, first + v.x, first + v.x + v.y, first + v.x + v.y + v.z);
        row_base += rows[q];
    }
    __syncthreads();
    return row_base - run;
}

__device__ __forceinline__ void zero_table(uint32_t *s_table) {
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q)
        reinterpret_cast<uint4 *>(s_table)[q * kThreads + threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
}

// Insertion sort of a short segment in shared memory (len <= kRegisterMax):
// few registers, and at a few particles per cell only a handful of steps.
__device__ __forceinline__ void insertion_sort_shared(uint32_t *seg, uint32_t len) {
    for (uint32_t i = 1; i < len; ++i) {
        const uint32_t x = seg[i];
        uint32_t j = i;
        for (; j > 0 && seg[j - 1] > x; --j) seg[j] = seg[j - 1];
        seg[j] = x;
    }
}

// Phase 2 for a bucket of at most kHeld particles: its pairs held in shared
// memory, placed in s_order, then ordenado and destino written in order.
template <bool kStable>
__device__ __forceinline__ void held_bucket(const SparseArgs &a, uint64_t cell_lo, uint64_t cell_hi, uint32_t base,
                                            uint32_t total, uint32_t ctas, uint32_t *s_table, uint2 *s_pair,
                                            uint32_t *s_slot, uint32_t *s_order, const uint32_t *s_off,
                                            const uint32_t *s_src, uint32_t (*s_rows)[kWarps], uint2 *s_long,
                                            uint32_t *s_nlong) {
    const uint32_t tid = threadIdx.x;
    for (uint32_t k = tid; k < total; k += kThreads) {
        const uint32_t s = source_of(s_off, ctas, k);
        const uint2 pr = a.pairs[s_src[s] + (k - s_off[s])];
        s_pair[k] = make_uint2(pr.x - (uint32_t)cell_lo, pr.y);
    }
    __syncthreads();
    uint32_t run = 0;  // bucket-local position of the window's first particle
    for (uint64_t w0 = cell_lo; w0 < cell_hi; w0 += kWindow) {
        const uint32_t wl = (uint32_t)(w0 - cell_lo), win = (uint32_t)min((uint64_t)kWindow, cell_hi - w0);
        zero_table(s_table);
        for (uint32_t k0 = 0; k0 < total; k0 += kThreads) {
            const uint32_t k = k0 + tid;
            const uint32_t c = k < total ? s_pair[k].x - wl : 0u;
            const bool mine = k < total && c < win;
            const uint32_t slot = smem_take(s_table, mine, c);
            if (mine) s_slot[k] = slot;
        }
        __syncthreads();
        const uint32_t wtotal = scan_window(a.conteos, a.inicios, s_table, w0, cell_hi, run, base, s_rows);
        for (uint32_t k = tid; k < total; k += kThreads) {
            const uint2 pr = s_pair[k];
            const uint32_t c = pr.x - wl;
            if (c < win) s_order[s_table[c] + s_slot[k]] = pr.y;
        }
        __syncthreads();
        if constexpr (kStable) {
            // Short segments now; long ones once every window is placed.
            for (uint32_t c = tid; c < win; c += kThreads) {
                const uint32_t st = s_table[c], en = c + 1 < win ? s_table[c + 1] : run + wtotal;
                if (en - st > (uint32_t)kRegisterMax) {
                    const uint32_t q = atomicAdd(s_nlong, 1u);
                    if (q < kLongMax) s_long[q] = make_uint2(st, en - st);  // total / 33 < kLongMax
                } else if (en - st > 1) {
                    insertion_sort_shared(s_order + st, en - st);
                }
            }
        }
        run += wtotal;
        __syncthreads();
    }
    if constexpr (kStable) {
        uint32_t *s_buf = reinterpret_cast<uint32_t *>(s_pair);  // 2 * kHeld words, free now
        const uint32_t nlong = min(*s_nlong, kLongMax);
        for (uint32_t q = 0; q < nlong; ++q) {
            const uint2 seg = s_long[q];
            for (uint32_t i = tid; i < seg.y; i += kThreads) s_buf[i] = s_order[seg.x + i];
            bitonic_shared<kThreads>(s_buf, seg.y);
            for (uint32_t i = tid; i < seg.y; i += kThreads) s_order[seg.x + i] = s_buf[i];
            __syncthreads();
        }
    }
    for (uint32_t k = tid; k < total; k += kThreads) a.ordenado[base + k] = s_order[k];
    // destino: two threads per record, every load of a round before its stores
    constexpr uint32_t kHalves = 4;
    for (uint32_t h0 = 0; h0 < 2u * total; h0 += kHalves * kThreads) {
        uint4 v[kHalves];
#pragma unroll
        for (uint32_t e = 0; e < kHalves; ++e) {
            const uint32_t h = h0 + e * kThreads + tid;
            if (h < 2u * total) v[e] = load_nc_na(a.origen + 2 * (uint64_t)s_order[h >> 1] + (h & 1u));
        }
#pragma unroll
        for (uint32_t e = 0; e < kHalves; ++e) {
            const uint32_t h = h0 + e * kThreads + tid;
            if (h < 2u * total) store_cs(a.destino + 2 * (uint64_t)base + h, v[e]);
        }
    }
}

// Phase 2 for a bucket of more than kHeld particles (a crowded region): each
// window of cells reads the bucket's pairs from the workspace twice, to count
// and to place, and places them straight into ordenado.  In stable mode each
// cell's segment is then sorted where it lies and the window's records
// gathered after.  Out of line: it is rare, and its registers would weigh on
// the common path.
template <bool kStable>
__device__ __noinline__ void streamed_bucket(const uint4 *origen, uint4 *destino, uint32_t *conteos,
                                             uint32_t *inicios, uint32_t *ordenado, const uint2 *pairs,
                                             uint32_t *scratch, uint32_t n, uint64_t cell_lo, uint64_t cell_hi,
                                             uint32_t base, uint32_t total, uint32_t ctas, uint32_t *s_table,
                                             uint2 *s_pair, const uint32_t *s_off, const uint32_t *s_src,
                                             uint32_t (*s_rows)[kWarps], uint2 *s_long, uint32_t *s_nlong) {
    const uint32_t tid = threadIdx.x;
    uint32_t run = 0;
    for (uint64_t w0 = cell_lo; w0 < cell_hi; w0 += kWindow) {
        const uint32_t win = (uint32_t)min((uint64_t)kWindow, cell_hi - w0);
        zero_table(s_table);
        for (uint32_t k0 = 0; k0 < total; k0 += kThreads) {
            const uint32_t k = k0 + tid;
            uint32_t c = 0u;
            if (k < total) {
                const uint32_t s = source_of(s_off, ctas, k);
                c = pairs[s_src[s] + (k - s_off[s])].x - (uint32_t)w0;
            }
            smem_take(s_table, k < total && c < win, c);
        }
        __syncthreads();
        const uint32_t wtotal = scan_window(conteos, inicios, s_table, w0, cell_hi, run, base, s_rows);
        for (uint32_t k0 = 0; k0 < total; k0 += kThreads) {
            const uint32_t k = k0 + tid;
            uint2 pr = make_uint2(0u, 0u);
            if (k < total) {
                const uint32_t s = source_of(s_off, ctas, k);
                pr = pairs[s_src[s] + (k - s_off[s])];
            }
            const uint32_t c = pr.x - (uint32_t)w0;
            const bool mine = k < total && c < win;
            const uint32_t pos = smem_take(s_table, mine, c);
            if (mine) {
                ordenado[base + pos] = pr.y;
                if (!kStable) {
                    destino[2 * ((uint64_t)base + pos)] = load_nc_na(origen + 2 * (uint64_t)pr.y);
                    destino[2 * ((uint64_t)base + pos) + 1] = load_nc_na(origen + 2 * (uint64_t)pr.y + 1);
                }
            }
        }
        __syncthreads();
        if constexpr (kStable) {
            // s_table[c] is now the end of cell c's segment.  Cells in rounds
            // of kThreads, each round's long segments sorted by the whole CTA
            // in the pair buffer (unused on this path).
            for (uint32_t c0 = 0; c0 < win; c0 += kThreads) {
                const uint32_t c = c0 + tid;
                if (c < win) {
                    const uint32_t st = c == 0 ? run : s_table[c - 1], en = s_table[c];
                    if (en - st > 1 && !sort_short_segment(ordenado + base + st, en - st)) {
                        const uint32_t q = atomicAdd(s_nlong, 1u);
                        s_long[q] = make_uint2(st, en - st);  // at most one per thread
                    }
                }
                __syncthreads();
                const uint32_t nlong = *s_nlong;
                for (uint32_t q = 0; q < nlong; ++q) {
                    const uint2 seg = s_long[q];
                    sort_long_segment<kThreads>(ordenado + base + seg.x, scratch + base + seg.x, seg.y, n,
                                                reinterpret_cast<uint32_t *>(s_pair), 2 * kHeld);
                }
                __syncthreads();
                if (tid == 0) *s_nlong = 0u;
                __syncthreads();
            }
            for (uint64_t h = 2 * ((uint64_t)base + run) + tid; h < 2 * ((uint64_t)base + run + wtotal);
                 h += kThreads) {
                const uint32_t i = ordenado[h >> 1];
                destino[h] = load_nc_na(origen + 2 * (uint64_t)i + (h & 1u));
            }
        }
        run += wtotal;
        __syncthreads();
    }
}

template <bool kStable>
__global__ void __launch_bounds__(kThreads, 2) build_sparse_kernel(SparseArgs a, Geometry g, grid_ws_header *hdr) {
    extern __shared__ __align__(16) uint32_t s_dyn[];
    uint32_t *s_table = s_dyn;                                        // [kWindow] cell counts, then starts
    uint2 *s_pair = reinterpret_cast<uint2 *>(s_table + kWindow);     // [kHeld] (cell, particle)
    uint32_t *s_slot = reinterpret_cast<uint32_t *>(s_pair + kHeld);  // [kHeld] slot in the cell / bucket
    uint32_t *s_order = s_slot + kHeld;                               // [kHeld] cell, then the cell order
    __shared__ uint32_t s_hist[kThreads];  // phase 1: particles per bucket; phase 2: run starts
    __shared__ uint32_t s_src[kThreads];   // phase 2: first pair of each source's run
    __shared__ uint32_t s_red[kWarps];
    __shared__ uint2 s_red2[kWarps];
    __shared__ uint32_t s_rows[kScanVecs + 1][kWarps];
    __shared__ uint2 s_long[kStable ? kLongMax : 1];
    __shared__ uint32_t s_nlong;
    const uint32_t tid = threadIdx.x;
    const uint32_t ctas = gridDim.x;
    uint32_t passed = 0;

    // Phase 2 writes over the fused build's counter array (the table lives
    // there): a later build that uses it clears it first.
    if (blockIdx.x == 0 && tid == 0) {
        hdr->counts_clean = 0u;
        a.inicios[a.cells] = a.n;
    }
    s_hist[tid] = 0u;
    if (tid == 0) s_nlong = 0u;
    __syncthreads();

    // ---- phase 1: this CTA's particles, cells and buckets
    uint64_t p_lo, p_hi;
    fused::particle_range(a.n, p_lo, p_hi);
    const uint32_t m = (uint32_t)(p_hi - p_lo);
    for (uint32_t i0 = 0; i0 < m; i0 += kRoundItems * kThreads) {
        uint4 rec[kRoundItems];
#pragma unroll
        for (uint32_t k = 0; k < kRoundItems; ++k) {
            const uint32_t i = i0 + k * kThreads + tid;
            if (i < m) rec[k] = load_nc_na(a.origen + 2 * (p_lo + i));
        }
#pragma unroll
        for (uint32_t k = 0; k < kRoundItems; ++k) {
            const uint32_t i = i0 + k * kThreads + tid;
            const bool valid = i < m;
            const uint32_t c = valid ? cell_of(rec[k], g) : 0u;
            const uint32_t b = (uint32_t)__umul64hi((unsigned long long)c, a.magic);
            const uint32_t slot = smem_take(s_hist, valid, b);
            if (valid) {
                a.celdaDe[p_lo + i] = c;
                s_order[i] = c;
                s_slot[i] = slot;
            }
        }
    }
    __syncthreads();
    {
        // Row b of the table, column blockIdx.x: this CTA's particles in
        // buckets below b (row `buckets` holds them all).
        uint32_t total;
        const uint32_t excl = block_exclusive_scan(tid < a.buckets ? s_hist[tid] : 0u, s_red, &total);
        if (tid <= a.buckets) a.table[(uint64_t)tid * ctas + blockIdx.x] = excl;
        s_hist[tid] = excl;
    }
    __syncthreads();
    for (uint32_t i = tid; i < m; i += kThreads) {
        const uint32_t c = s_order[i];
        const uint32_t b = (uint32_t)__umul64hi((unsigned long long)c, a.magic);
        s_pair[s_hist[b] + s_slot[i]] = make_uint2(c, (uint32_t)p_lo + i);
    }
    __syncthreads();
    for (uint32_t i = tid; i < m; i += kThreads) a.pairs[p_lo + i] = s_pair[i];

    fused::grid_arrive(hdr, passed);
    // While the barrier fills: conteos of this CTA's bucket set to zero, so
    // that phase 2 writes only the counts that are not (most cells of a
    // sparse grid are empty, and these stores overlap the wait).
    if (blockIdx.x < a.buckets) {
        const uint64_t lo = (uint64_t)blockIdx.x * a.width, hi = min(a.cells, lo + a.width);
        uint4 *c4 = reinterpret_cast<uint4 *>(a.conteos + lo);
        const uint64_t quads = (hi - lo) / 4;
        for (uint64_t q = tid; q < quads; q += kThreads) c4[q] = make_uint4(0u, 0u, 0u, 0u);
        for (uint64_t c = lo + 4 * quads + tid; c < hi; c += kThreads) a.conteos[c] = 0u;
    }
    const bool complete = wait_all(hdr, passed, &s_red[0]);

    // ---- phase 2: this CTA's bucket (none after a wait that gave up: the
    // table may be incomplete)
    const uint32_t b = blockIdx.x;
    if (b < a.buckets && complete) {
        const uint64_t cell_lo = (uint64_t)b * a.width;
        const uint64_t cell_hi = min(a.cells, cell_lo + a.width);
        uint32_t base, total;
        {
            // Column b: where each source's run of this bucket starts, and
            // how many of its particles lie in lower buckets.
            uint32_t e0 = 0u, e1 = 0u;
            if (tid < ctas) {
                e0 = a.table[(uint64_t)b * ctas + tid];
                e1 = a.table[(uint64_t)(b + 1) * ctas + tid];
            }
            uint32_t off;
            pair_scan(e0, e1 - e0, s_red2, &base, &off, &total);
            if (tid < ctas) {
                s_hist[tid] = off;
                s_src[tid] = (uint32_t)((uint64_t)a.n * tid / ctas) + e0;
            }
            if (tid == 0) s_hist[ctas] = total;
        }
        __syncthreads();
        if (total <= kHeld)
            held_bucket<kStable>(a, cell_lo, cell_hi, base, total, ctas, s_table, s_pair, s_slot, s_order, s_hist,
                                 s_src, s_rows, s_long, &s_nlong);
        else
            streamed_bucket<kStable>(a.origen, a.destino, a.conteos, a.inicios, a.ordenado, a.pairs, a.scratch, a.n,
                                     cell_lo, cell_hi, base, total, ctas, s_table, s_pair, s_hist, s_src, s_rows,
                                     s_long, &s_nlong);
    }
    fused::leave_launch(hdr);
}

std::atomic<int> g_grid[2][kMaxDevices];  // cached grid size per mode and device (0 = not yet known)

template <bool kStable>
cudaError_t sparse_grid(int device, int *grid) {
    if (device >= 0 && device < kMaxDevices) {
        const int cached = g_grid[kStable][device].load(std::memory_order_relaxed);
        if (cached != 0) {
            *grid = cached;
            return cached > 0 ? cudaSuccess : cudaErrorNotSupported;
        }
    }
    int coop = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaFuncSetAttribute(build_sparse_kernel<kStable>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDynamicSmem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_sparse_kernel<kStable>, kThreads,
                                                          kDynamicSmem);
    if (e != cudaSuccess) return e;
    int gsz = coop ? per_sm * sms : -1;
    // A table row per bucket and a scan over the sources need fewer CTAs
    // than threads per CTA.
    if (gsz <= 0 || gsz >= kThreads) gsz = -1;
    if (device >= 0 && device < kMaxDevices) g_grid[kStable][device].store(gsz, std::memory_order_relaxed);
    *grid = gsz;
    return gsz > 0 ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_build_sparse(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n, uint64_t cells,
                                const Geometry &g, grid_ws_header *hdr, uint32_t *counts, uint32_t *pairs,
                                bool stable, uint32_t *sort_scratch, cudaStream_t s) {
    int device = 0, grid = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = stable ? sparse_grid<true>(device, &grid) : sparse_grid<false>(device, &grid);
    if (e != cudaSuccess) return e;
    // Every CTA's particles fit its pair buffer; one bucket per CTA, of a
    // width that keeps 16-byte stores aligned; the table fits the counters.
    if (n == 0 || (uint64_t)n > (uint64_t)grid * kSparseMaxParticlesPerCta) return cudaErrorNotSupported;
    uint64_t w = (cells + (uint64_t)grid - 1) / (uint64_t)grid;
    w = (w + 3) & ~3ull;
    const uint64_t buckets = (cells + w - 1) / w;
    if (w > 0xffffffffull || (buckets + 1) * (uint64_t)grid > cells) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDynamicSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const SparseArgs a{reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino), conteos, celdaDe,
                       inicios, ordenado, reinterpret_cast<uint2 *>(pairs), counts, sort_scratch, n, cells,
                       (uint32_t)w, (uint32_t)buckets, ~0ull / w + 1ull};
    return cudaLaunchKernelEx(&cfg, stable ? build_sparse_kernel<true> : build_sparse_kernel<false>, a, g, hdr);
}

}  // namespace ugrid
