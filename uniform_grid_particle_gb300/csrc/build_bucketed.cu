// The grid build as a two-level counting sort, in one cooperative launch.
//
// The pages count with one global atomic per particle ("Contar partículas por
// celda", §El kernel).  With about one particle per cell nothing can be
// grouped, and the L2 atomic units become the limit of the whole build.  This
// build reaches the same outputs with atomics in shared memory, plus one
// global atomic per CTA and bucket, by first sorting the particles into
// buckets of `width` consecutive cells (as in the first pass of an MSD radix
// sort):
//
//   A  cells: celdaDe[i] = cell of particle i; each CTA histograms its
//      particles over the buckets in shared memory and adds its histogram to
//      the bucket totals, one global atomic per CTA and bucket, whose old
//      value is where the CTA's stretch of the bucket starts
//   C  bucket bases = exclusive scan of the totals; each CTA sends its
//      particles to its stretches as (cell, particle) pairs
//   D  per bucket, one CTA: a shared-memory histogram over the bucket's cells
//      gives conteos and, scanned from the bucket's base, inicios ("Construir
//      el índice de la rejilla con un prefix sum", §Del conteo al inicio);
//      the slot each particle took in its cell's counter places it
//      (§La dispersión), and the bucket's stretch of ordenado and destino is
//      written in order ("Reordenar por celda…", §El kernel de reordenación:
//      destino[k] = origen[ordenado[k]])
//
// Every output is one the pages' chain can produce: conteos and inicios are
// the histogram and its exclusive scan, and each cell's segment of ordenado
// holds exactly its particles (in shared-memory arrival order).
//
// The buckets are `width` consecutive cells (a multiple of 4, so bucket
// boundaries keep 16-byte alignment); the bucket of cell c is c / width,
// taken as the high word of c * ceil(2^64 / width), exact for every 32-bit c
// because c * (ceil(2^64 / width) * width - 2^64) < 2^32 * width < 2^64.
// The plan makes the bucket count a multiple of the CTA count, so in a
// uniform scene every CTA places the same number of buckets.
//
// A bucket's total is kBucketLanes words, CTA j adding to lane
// j mod kBucketLanes: a word then takes the atomics of only
// ctas / kBucketLanes CTAs (atomics on one word are serialised in L2).  Lane
// r's part of a bucket starts after the totals of lanes 0..r-1.  The totals
// are zero between builds: the CTA that places a bucket zeroes its words, and
// a header word records that all of them are clean (a build that did not
// finish leaves it unset and the next one clears them first).
//
// A bucket of more than kBucketCap particles would not fit one CTA's shared
// memory.  Every CTA sees the same totals, so all of them then take the
// atomic path of the fused build instead (count from celdaDe, scan, scatter
// with the records), and the result is the same.
//
// Phases A and C read a CTA's contiguous range of particles, phase D takes
// buckets cyclically, and grid barriers separate the phases (see
// fused_common.cuh: bounded waits that record kStatusTimeout).
#include <atomic>

#include "fused_common.cuh"

namespace ugrid {
namespace {

using namespace fused;

constexpr int kBucketItems = (int)(kBucketCap / kThreads);  // particles per thread in phase D
static_assert(kBucketItems * kThreads == (int)kBucketCap, "phase D takes a whole bucket in one round");
static_assert(kBucketMaxCells == kScanVecs * 4 * kThreads && kBucketMaxCount == kScanVecs * 4 * kThreads,
              "bucket tables are the 32 KB scan table");
constexpr size_t kTableBytes = (size_t)kScanVecs * kThreads * sizeof(uint4);  // 32 KB
constexpr size_t kDynamicSmem = kTableBytes + 3 * kBucketCap * sizeof(uint32_t);  // + 3 x 16 KB buffers
constexpr uint32_t kCacheMax = 6144;  // particles per CTA whose cell and rank phase A keeps for phase C
static_assert(2 * kCacheMax <= 3 * kBucketCap, "phase A's cache fits the three buffers");
constexpr int kMaxDevices = 64;
// Stable mode: cells of one bucket longer than kRegisterMax particles; at most
// kBucketCap / (kRegisterMax + 1) of them fit in a bucket.
constexpr uint32_t kLongMax = kBucketCap / (kRegisterMax + 1) + 1;
// The first buckets a CTA places: phase C keeps their bases and sizes in
// shared memory (any others are read back from the workspace).
constexpr uint32_t kOwnMax = 32;
// Phase D's gather: records per warp chunk (four per lane) and the stage bytes.
constexpr uint32_t kGatherChunk = 128;
constexpr uint32_t kStageBytes = kGatherChunk * sizeof(ugrid_particula);
static_assert((kWarps / 2) * kStageBytes <= kTableBytes && (kWarps / 2) * kStageBytes <= 2 * kBucketCap * 4,
              "half the warps stage in the cell table, half in the slot buffers");

struct BucketScratch {
    uint32_t width;              // cells per bucket
    uint32_t buckets;            // B
    unsigned long long magic;    // ceil(2^64 / width)
    uint32_t *total;             // [B][kBucketLanes] particles per bucket and lane, zero between builds
    uint32_t *base;              // [B] first position of each bucket
    uint2 *pairs;                // [n] (cell, particle), grouped by bucket
};

__device__ __forceinline__ uint32_t bucket_of(uint32_t c, const BucketScratch &bk) {
    return (uint32_t)__umul64hi((unsigned long long)c, bk.magic);
}

static_assert(kBucketLanes == 8, "a bucket's lane words are two 16-byte vectors");

// Particles of bucket b (all lanes) and, in `before`, those of lanes below r.
__device__ __forceinline__ uint32_t bucket_total(const uint32_t *total, uint32_t b, uint32_t r, uint32_t &before) {
    const uint4 *p = reinterpret_cast<const uint4 *>(total + (uint64_t)b * kBucketLanes);
    const uint4 lo = p[0], hi = p[1];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t sum = 0, pre = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        pre += (uint32_t)e < r ? w[e] : 0u;
        sum += w[e];
    }
    before = pre;
    return sum;
}

__device__ __forceinline__ void zero_bucket(uint32_t *total, uint32_t b) {
    uint4 *t = reinterpret_cast<uint4 *>(total + (uint64_t)b * kBucketLanes);
    t[0] = t[1] = make_uint4(0u, 0u, 0u, 0u);
}

// Phase D's record move for one bucket (destino[base + q] = origen[s_order[q]],
// q < t): each warp takes chunks of 128 positions; every lane names four rows
// in one tile::gather4 copy into the warp's 4 KB stage, the warp's mbarrier
// counts them in, and one bulk copy writes the chunk to destino.  A chunk
// whose rows lie close together is read with 16-byte loads instead.  A
// chunk naming a row >= n is copied with plain loads, without that row, and
// sets the bounds bit.  `uses` counts the phases of the warp's mbarrier.
__device__ __forceinline__ void gather_bucket(const CUtensorMap *map, const BuildArgs &a, const uint32_t *s_order,
                                              uint32_t t, uint32_t base, unsigned char *stage, uint32_t bar,
                                              uint32_t &uses, uint32_t *status) {
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t chunks = (t + kGatherChunk - 1u) / kGatherChunk;
    for (uint32_t c = warp; c < chunks; c += kWarps) {
        const uint32_t c0 = c * kGatherChunk, rows = min(kGatherChunk, t - c0);
        const uint32_t q0 = c0 + 4u * lane;
        const uint32_t v = q0 < t ? min(4u, t - q0) : 0u;
        int row[4] = {0, 0, 0, 0};
        bool lane_bad = false;
        if (v > 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t r = s_order[q0 + min((uint32_t)e, v - 1u)];
                lane_bad |= r >= a.n;
                row[e] = (int)r;
            }
        }
        uint4 *dst = a.destino + 2 * ((uint64_t)base + c0);
        if (__any_sync(0xffffffffu, lane_bad)) {
            if (lane_bad) record_status(status, kStatusBounds);
            for (uint32_t h = lane; h < 2u * rows; h += 32u) {
                const uint32_t src = s_order[c0 + (h >> 1)];
                if (src < a.n) store_cs(dst + h, load_nc_na(a.origen + 2 * (uint64_t)src + (h & 1u)));
            }
            continue;
        }
        if (rows_span(row, v) < kClusterRows) {
            // Rows close together (input already near cell order): 16-byte
            // loads share their lines; four in flight per lane.
            for (uint32_t h0 = 0; h0 < 2u * rows; h0 += 4u * 32u) {
                uint4 r4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t h = h0 + (uint32_t)k * 32u + lane;
                    if (h < 2u * rows)
                        r4[k] = load_nc_na(a.origen + 2 * (uint64_t)s_order[c0 + (h >> 1)] + (h & 1u));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t h = h0 + (uint32_t)k * 32u + lane;
                    if (h < 2u * rows) store_cs(dst + h, r4[k]);
                }
            }
            continue;
        }
        const uint32_t lanes = __popc(__ballot_sync(0xffffffffu, v > 0));
        if (lane == 0) mbar_arrive_expect(bar, lanes * 4u * (uint32_t)sizeof(ugrid_particula));
        __syncwarp();
        if (v > 0) gather4_records(smem_addr(stage + 4u * lane * sizeof(ugrid_particula)), map, row, bar);
        if (!__all_sync(0xffffffffu, mbar_wait(bar, uses & 1u))) {  // the warp agrees on a timeout
            if (lane == 0) record_status(status, kStatusTimeout);
            return;
        }
        ++uses;
        if (lane == 0) bulk_store_wait_read(dst, smem_addr(stage), rows * (uint32_t)sizeof(ugrid_particula));
        __syncwarp();
    }
}

// Bands for pairs_from_celdaDe.  Each stretch a CTA writes keeps about two
// partly written 128-byte lines open (its first and its last) until it is
// full; with every CTA's stretches like this one's (`touched` buckets),
// enough bands that one band's open lines take at most kBandBytes of L2.
// Input already in cell order touches few buckets per CTA: one band.
constexpr uint64_t kBandBytes = 96ull << 20;
__device__ __forceinline__ uint32_t pair_bands(uint32_t touched, uint32_t ctas) {
    const uint64_t open = (uint64_t)ctas * touched * 2 * 128;
    const uint64_t bands = (open + kBandBytes - 1) / kBandBytes;
    return (uint32_t)max((uint64_t)1, min(bands, (uint64_t)64));
}

// Phase C's pairs when phase A could not keep the CTA's cells and ranks
// (more particles per CTA than its cache holds): cells re-read from celdaDe,
// places taken from the shared cursors.  The writes are scattered 8-byte
// stores into every CTA's stretch of every bucket; when those stretches are
// too many for their partly written lines to stay in L2 until they fill,
// the lines go to DRAM half written.  So the buckets are taken in `bands`
// passes of consecutive buckets, each pass re-reading celdaDe and writing
// only the pairs of its band: a band's open lines fit in L2.  Out of line:
// on the common sizes it never runs, and its code stays out of the way of
// the code that does.
__device__ __noinline__ void pairs_from_celdaDe(const BuildArgs a, const BucketScratch bk, uint32_t *s_table,
                                                uint64_t p_lo, uint64_t p_hi, uint32_t bands, uint32_t *status) {
    const uint32_t per_band = (bk.buckets + bands - 1) / bands;
    for (uint32_t band = 0; band < bands; ++band) {
        const uint32_t b_lo = band * per_band, b_hi = min(bk.buckets, b_lo + per_band);
        for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kScatterItems) {
            uint32_t cell[kScatterItems];
#pragma unroll
            for (int k = 0; k < kScatterItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + threadIdx.x;
                if (i < p_hi) cell[k] = a.celdaDe[i];
            }
#pragma unroll
            for (int k = 0; k < kScatterItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + threadIdx.x;
                const uint32_t b = i < p_hi ? bucket_of(cell[k], bk) : 0u;
                const bool valid = i < p_hi && b >= b_lo && b < b_hi;
                const uint32_t q = smem_take(s_table, valid, valid ? b : 0u);
                if (valid) {
                    if (q < a.n)
                        bk.pairs[q] = make_uint2(cell[k], (uint32_t)i);
                    else
                        record_status(status, kStatusBounds);
                }
            }
        }
    }
}

// A bucket too large for one CTA: every CTA takes the atomic path of the
// fused build from celdaDe on (with its stable tail in stable mode).  Kept out
// of line so that its registers do not weigh on the bucketed phases.
template <bool kStable>
__device__ __noinline__ void atomic_path(const BuildArgs a, const Geometry g, grid_ws_header *hdr,
                                         const FusedScratch ws, const BucketScratch bk, bool clean,
                                         uint32_t &passed, uint64_t p_lo, uint64_t p_hi, uint4 (*s_held)[kThreads],
                                         uint32_t *s_red, uint32_t (*s_rows)[kWarps]) {
    if (!clean) {
        clear_counters(ws.counts, a.cells);
        grid_barrier(hdr, passed);
    }
    count_phase<false>(a, g, ws, p_lo, p_hi, s_held);
    grid_barrier(hdr, passed);
    if (blockIdx.x == 0 && threadIdx.x == 0) hdr->counts_clean = 0u;
    // Every CTA has read the bucket totals by now: clear them for the next build.
    for (uint32_t b = blockIdx.x * kThreads + threadIdx.x; b < bk.buckets; b += gridDim.x * kThreads)
        zero_bucket(bk.total, b);
    const ScanChunk chunk = scan_chunk(a.cells);
    scan_totals_phase(ws, chunk, s_held, s_red);
    grid_barrier(hdr, passed);
    scan_starts_phase(a, ws, chunk, s_held, s_red, s_rows);
    grid_barrier(hdr, passed);
    if (blockIdx.x == 0 && threadIdx.x == 0 && (hdr->status & kStatusTimeout) == 0)
        hdr->counts_clean = (uint32_t)a.cells;
    if constexpr (kStable)
        stable_tail_phase(a, ws, hdr, passed, p_lo, p_hi, s_held);
    else
        scatter_move_phase(a, ws, &hdr->status, p_lo, p_hi);
}

template <bool kStable>
__global__ void __launch_bounds__(kThreads, 2)
build_bucketed_kernel(const __grid_constant__ CUtensorMap origen_map, BuildArgs a, Geometry g, grid_ws_header *hdr,
                      FusedScratch ws, BucketScratch bk) {
    extern __shared__ __align__(1024) uint4 s_dyn[];
    uint4(*s_held)[kThreads] = reinterpret_cast<uint4(*)[kThreads]>(s_dyn);
    uint32_t *s_table = reinterpret_cast<uint32_t *>(s_dyn);                        // u32[8192], same bytes
    uint32_t *s_order = reinterpret_cast<uint32_t *>(s_dyn + kScanVecs * kThreads);  // u32[kBucketCap]
    uint32_t *s_who = s_order + kBucketCap;                                           // u32[kBucketCap]
    uint32_t *s_place = s_who + kBucketCap;                                           // u32[kBucketCap]
    uint32_t *s_cell = s_order, *s_rank = s_order + kCacheMax;  // phase A's cache, over the three buffers
    __shared__ uint32_t s_red[kWarps];
    __shared__ uint32_t s_rows[kScanVecs + 1][kWarps];  // + the rows' totals
    __shared__ uint32_t s_clean, s_bclean, s_base, s_count, s_nlong;
    __shared__ uint32_t s_touched;  // buckets this CTA has particles in
    __shared__ uint32_t s_own_base[kOwnMax], s_own_count[kOwnMax];
    __shared__ __align__(8) unsigned long long s_gbar[kWarps];  // one per warp, phase D's gather
    __shared__ uint32_t s_long[kLongMax];  // stable mode: cells of the bucket with more than 32 particles
    // Stable mode: cells of the bucket with two particles or more (the only
    // segments to sort), listed by the particle that takes slot 1.
    __shared__ uint32_t s_multi[kStable ? kBucketCap / 2 : 1];
    __shared__ uint32_t s_nmulti;
    const uint32_t tid = threadIdx.x;
    const uint32_t ctas = gridDim.x;
    const uint32_t B = bk.buckets;
    uint32_t passed = 0;
    if (tid == 0) {
        s_clean = *reinterpret_cast<volatile uint32_t *>(&hdr->counts_clean) >= a.cells;
        s_bclean = *reinterpret_cast<volatile uint32_t *>(&hdr->buckets_clean) != 0u;
        s_touched = 0u;
    }
#pragma unroll
    for (int q = 0; q < kScanVecs; ++q) s_held[q][tid] = make_uint4(0u, 0u, 0u, 0u);  // s_table, 8192 words
    if ((tid & 31u) == 0) mbar_init(smem_addr(&s_gbar[tid >> 5]));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    uint32_t gather_uses = 0;  // phases of this warp's gather mbarrier
    // Nobody touches the long-segment queue of the atomic path before its stable tail.
    if (kStable && blockIdx.x == 0 && tid == 0) hdr->stable_big = 0u;
    __syncthreads();
    uint64_t p_lo, p_hi;
    particle_range(a.n, p_lo, p_hi);
    const uint32_t mine = (uint32_t)(p_hi - p_lo);
    const bool cached = mine <= kCacheMax;
    // Phase C can then write the pairs bucket by bucket (runs of consecutive
    // positions) when the table has room for a second copy of the histogram
    // and for the CTA's particles in bucket order.
    const bool grouped = cached && B <= 4u * kThreads && 2u * B + mine <= kBucketMaxCount;

    if (!s_bclean) {
        for (uint32_t b = blockIdx.x * kThreads + tid; b < B; b += ctas * kThreads) zero_bucket(bk.total, b);
        grid_barrier(hdr, passed);
    }

    // ---- A: cells and the bucket totals ------------------------------------------
    {
        unsigned long long keep;
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
        for (uint64_t r0 = p_lo; r0 < p_hi; r0 += (uint64_t)kThreads * kCountItems) {
            uint4 rec[kCountItems];
#pragma unroll
            for (int k = 0; k < kCountItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                if (i < p_hi) rec[k] = load_policy(a.origen + 2 * i, keep);
            }
#pragma unroll
            for (int k = 0; k < kCountItems; ++k) {
                const uint64_t i = r0 + (uint64_t)k * kThreads + tid;
                const bool valid = i < p_hi;
                uint32_t bucket = 0u, c = 0u;
                if (valid) {
                    c = cell_of(rec[k], g);
                    a.celdaDe[i] = c;
                    bucket = bucket_of(c, bk);
                }
                const uint32_t rank = smem_take(s_table, valid, bucket);
                if (valid && cached) {
                    s_cell[i - p_lo] = c;
                    s_rank[i - p_lo] = rank;
                }
            }
        }
    }
    __syncthreads();
    // This CTA's stretch within its lane of every bucket it has particles in:
    // the atomic's old value is the offset, and the lane words end as totals.
    uint32_t touched = 0;
    for (uint32_t b = tid; b < B; b += kThreads) {
        const uint32_t m = s_table[b];
        if (grouped) s_table[B + b] = m;  // the histogram, kept for phase C
        if (m) s_table[b] = atomicAdd(bk.total + (uint64_t)b * kBucketLanes + blockIdx.x % kBucketLanes, m);
        touched += m != 0u;
    }
    if (!cached && touched) atomicAdd(&s_touched, touched);
    grid_arrive(hdr, passed);
    if (grouped) {
        // Phase C writes this CTA's pairs as runs of consecutive positions,
        // one run per bucket, rather than one scattered 8-byte write per
        // particle: the CTA's particles in bucket order (its histogram
        // scanned, plus each particle's rank in its bucket).  This needs no
        // other CTA, so it runs while the barrier fills.
        uint32_t *s_from = s_table + B, *s_stage = s_table + 2u * B;
        {
            uint32_t h[kScanVecs], excl[kScanVecs], rows[kScanVecs];
            const uint32_t b0 = 4u * tid;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = b0 + e < B ? s_from[b0 + e] : 0u;
            h[0] = w[0] + w[1] + w[2] + w[3];
#pragma unroll
            for (int q = 1; q < kScanVecs; ++q) h[q] = 0u;
            rows_exclusive_scan<1>(h, excl, rows, s_rows);
            uint32_t f = excl[0];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (b0 + e < B) s_from[b0 + e] = f;
                f += w[e];
            }
        }
        __syncthreads();
        for (uint32_t k = tid; k < mine; k += kThreads) {
            const uint32_t at = s_from[bucket_of(s_cell[k], bk)] + s_rank[k];
            if (at < mine)
                s_stage[at] = k;
            else
                record_status(&hdr->status, kStatusBounds);
        }
    }
    grid_wait(hdr, passed);
    if (blockIdx.x == 0 && tid == 0) hdr->buckets_clean = 0u;

    // ---- C: bucket bases, this CTA's stretch of each bucket, the pairs ------------
    bool heavy;
    {
        const uint32_t lane_r = blockIdx.x % kBucketLanes;
        uint4 v[kScanVecs];
        uint32_t t[kScanVecs], most = 0;
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) {
            const uint32_t b0 = 4u * (q * kThreads + tid);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[e] = 0u;
                if (b0 + e < B) {
                    uint32_t before;
                    w[e] = bucket_total(bk.total, b0 + e, lane_r, before);
                    s_table[b0 + e] += before;  // this thread's own bucket: no other thread touches it
                }
            }
            v[q] = make_uint4(w[0], w[1], w[2], w[3]);
            t[q] = v[q].x + v[q].y + v[q].z + v[q].w;
            most = max(most, max(max(v[q].x, v[q].y), max(v[q].z, v[q].w)));
        }
        most = __reduce_max_sync(0xffffffffu, most);
        if (lane_id() == 0) s_red[tid >> 5] = most;
        uint32_t excl[kScanVecs], rows[kScanVecs];
        // its barriers also publish s_red; up to 4 * kThreads buckets fill one row
        if (B <= 4u * kThreads)
            rows_exclusive_scan<1>(t, excl, rows, s_rows);
        else
            rows_exclusive_scan(t, excl, rows, s_rows);
        most = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) most = max(most, s_red[w]);
        heavy = most > kBucketCap;
        if (!heavy) {
            uint32_t row_base = 0;
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) {
                const uint32_t b0 = 4u * (q * kThreads + tid);
                const uint32_t f = row_base + excl[q];
                const uint32_t start[4] = {f, f + v[q].x, f + v[q].x + v[q].y, f + v[q].x + v[q].y + v[q].z};
                const uint32_t size[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (b0 + e < B) {
                        if (blockIdx.x == 0) bk.base[b0 + e] = start[e];
                        s_table[b0 + e] += start[e];  // cursor of this CTA's stretch
                    }
                }
                // The buckets this CTA places in phase D, blockIdx.x + j * ctas:
                // their bases and sizes, from the thread that holds them.
                if (B <= 4u * kThreads) {
                    // One row of buckets: the thread that holds bucket bj.
                    if (q == 0) {
                        for (uint32_t j = 0, bj = blockIdx.x; bj < B && j < kOwnMax; ++j, bj += ctas) {
                            if ((bj >> 2) == tid) {
                                const uint32_t e = bj & 3u;
                                s_own_base[j] = e == 0 ? start[0] : e == 1 ? start[1] : e == 2 ? start[2] : start[3];
                                s_own_count[j] = e == 0 ? size[0] : e == 1 ? size[1] : e == 2 ? size[2] : size[3];
                            }
                        }
                    }
                } else if (b0 < B && ctas >= 4u) {
                    // Several rows: at most one of this thread's four buckets
                    // is one this CTA places (ctas >= 4 apart).
                    const uint32_t jj = b0 + 3u >= blockIdx.x ? (b0 + 3u - blockIdx.x) / ctas : kOwnMax;
                    const uint32_t bj = blockIdx.x + jj * ctas;
                    if (jj < kOwnMax && bj >= b0 && bj < b0 + 4u && bj < B) {
                        const uint32_t e = bj - b0;
                        s_own_base[jj] = e == 0 ? start[0] : e == 1 ? start[1] : e == 2 ? start[2] : start[3];
                        s_own_count[jj] = e == 0 ? size[0] : e == 1 ? size[1] : e == 2 ? size[2] : size[3];
                    }
                }
                row_base += rows[q];
            }
        }
    }
    __syncthreads();

    if (heavy) {
        atomic_path<kStable>(a, g, hdr, ws, bk, s_clean != 0u, passed, p_lo, p_hi, s_held, s_red, s_rows);
    } else {
        if (grouped) {
            const uint32_t *s_from = s_table + B, *s_stage = s_table + 2u * B;
            for (uint32_t j = tid; j < mine; j += kThreads) {
                const uint32_t k = s_stage[j];
                if (k >= mine) continue;
                const uint32_t c = s_cell[k], b = bucket_of(c, bk);
                const uint32_t q = s_table[b] + (j - s_from[b]);
                if (q < a.n)
                    bk.pairs[q] = make_uint2(c, (uint32_t)(p_lo + k));
                else
                    record_status(&hdr->status, kStatusBounds);
            }
        } else if (cached) {
            // Phase A kept each particle's cell and its rank among this CTA's
            // particles of its bucket: the pair's place needs no atomic.
            for (uint32_t k = tid; k < mine; k += kThreads) {
                const uint32_t c = s_cell[k];
                const uint32_t q = s_table[bucket_of(c, bk)] + s_rank[k];
                if (q < a.n)
                    bk.pairs[q] = make_uint2(c, (uint32_t)(p_lo + k));
                else
                    record_status(&hdr->status, kStatusBounds);
            }
        } else {
            pairs_from_celdaDe(a, bk, s_table, p_lo, p_hi, pair_bands(s_touched, ctas), &hdr->status);
        }
        grid_arrive(hdr, passed);
        // The first bucket's cell table is cleared while the barrier fills.
#pragma unroll
        for (int q = 0; q < kScanVecs; ++q) s_held[q][tid] = make_uint4(0u, 0u, 0u, 0u);
        grid_wait(hdr, passed);

        // ---- D: each bucket placed by one CTA ---------------------------------
        for (uint32_t b = blockIdx.x, j = 0; b < B; b += ctas, ++j) {
            const uint64_t cl = (uint64_t)b * bk.width;
            const uint32_t w = (uint32_t)min((uint64_t)bk.width, a.cells - cl);
            if (tid == 0) {
                s_nlong = 0u;
                s_nmulti = 0u;
                if (j < kOwnMax && (B <= 4u * kThreads || ctas >= 4u)) {
                    s_base = s_own_base[j];
                    s_count = s_own_count[j];
                } else {
                    s_base = bk.base[b];
                    uint32_t unused;
                    s_count = bucket_total(bk.total, b, 0u, unused);
                }
                zero_bucket(bk.total, b);  // clean for the next build
                // The next bucket's pairs, into L2 while this one is placed.
                if (j + 1 < kOwnMax && b + ctas < B && (B <= 4u * kThreads || ctas >= 4u)) {
                    const uint32_t nb = s_own_base[j + 1], nc = min(s_own_count[j + 1], kBucketCap);
                    if (nb <= a.n && nc <= a.n - nb && nc != 0u)
                        bulk_prefetch_l2(bk.pairs + nb, nc * (uint32_t)sizeof(uint2));
                }
            }
            __syncthreads();
            const uint32_t base = s_base;
            const uint32_t t = base <= a.n ? min(min(s_count, kBucketCap), a.n - base) : 0u;
            // (cell within the bucket) << 16 | slot within the cell; ~0u for none
            static_assert(kBucketItems % 4 == 0, "pairs loaded four at a time");
            uint2 prs[4];  // each group of four pairs is loaded before its first take
#pragma unroll
            for (int k = 0; k < kBucketItems; ++k) {
                if (k % 4 == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t qe = (uint32_t)(k + e) * kThreads + tid;
                        if (qe < t) prs[e] = bk.pairs[base + qe];
                    }
                }
                const uint32_t q = (uint32_t)k * kThreads + tid;
                bool valid = q < t;
                uint32_t local = 0u;
                if (valid) {
                    const uint2 pr = prs[k % 4];
                    local = pr.x - (uint32_t)cl;
                    s_who[q] = pr.y;
                    if (local >= w) {
                        record_status(&hdr->status, kStatusBounds);
                        valid = false;
                    }
                }
                const uint32_t slot = smem_take(s_table, valid, valid ? local : 0u);
                if (q < t) s_place[q] = valid ? (local << 16) | slot : 0xffffffffu;
                if (kStable && valid && slot == 1u) {
                    const uint32_t m = atomicAdd(&s_nmulti, 1u);
                    if (m < kBucketCap / 2) s_multi[m] = local;
                }
            }
            __syncthreads();
            {
                uint4 v[kScanVecs];
                uint32_t tt[kScanVecs], excl[kScanVecs], rows[kScanVecs];
#pragma unroll
                for (int q = 0; q < kScanVecs; ++q) {
                    v[q] = s_held[q][tid];
                    tt[q] = v[q].x + v[q].y + v[q].z + v[q].w;
                }
                rows_exclusive_scan(tt, excl, rows, s_rows);
                uint32_t row_base = base;
#pragma unroll
                for (int q = 0; q < kScanVecs; ++q) {
                    const uint64_t l = 4ull * (q * kThreads + tid);
                    const uint32_t f = row_base + excl[q];
                    store_starts(a.inicios + cl, l, w, f, v[q]);
                    if (l + 4 <= w) {
                        *reinterpret_cast<uint4 *>(a.conteos + cl + l) = v[q];
                    } else {
                        const uint32_t c3[3] = {v[q].x, v[q].y, v[q].z};
                        for (int e = 0; e < 3; ++e)
                            if (l + e < w) a.conteos[cl + l + e] = c3[e];
                    }
                    s_held[q][tid] = make_uint4(f, f + v[q].x, f + v[q].x + v[q].y, f + v[q].x + v[q].y + v[q].z);
                    row_base += rows[q];
                }
            }
            __syncthreads();
            for (uint32_t q = tid; q < t; q += kThreads) {
                const uint32_t place = s_place[q];
                if (place != 0xffffffffu) {
                    const uint32_t at = s_table[place >> 16] + (place & 0xffffu) - base;
                    if (at < t)
                        s_order[at] = s_who[q];
                    else
                        record_status(&hdr->status, kStatusBounds);
                }
            }
            __syncthreads();
            if constexpr (kStable) {
                // Every cell's segment of the bucket sorted by particle index
                // ("Construir el índice…", §El orden dentro de la celda):
                // short ones by one thread in registers, the rest by the whole
                // CTA, one at a time, in shared memory.  Only the cells of two
                // particles or more are visited.
                const uint32_t nmulti = min(s_nmulti, kBucketCap / 2);
                for (uint32_t i = tid; i < nmulti; i += kThreads) {
                    const uint32_t l = s_multi[i];
                    const uint32_t s0 = s_table[l] - base, e0 = (l + 1 < w ? s_table[l + 1] : base + t) - base;
                    if (e0 > s0 + 1 && e0 <= t && !sort_short_segment(s_order + s0, e0 - s0)) {
                        const uint32_t q = atomicAdd(&s_nlong, 1u);
                        if (q < kLongMax)
                            s_long[q] = l;
                        else
                            record_status(&hdr->status, kStatusBounds);
                    }
                }
                __syncthreads();
                const uint32_t nlong = min(s_nlong, kLongMax);
                for (uint32_t q = 0; q < nlong; ++q) {
                    const uint32_t l = s_long[q];
                    const uint32_t s0 = s_table[l] - base, e0 = (l + 1 < w ? s_table[l + 1] : base + t) - base;
                    for (uint32_t i = tid; i < e0 - s0; i += kThreads) s_who[i] = s_order[s0 + i];
                    bitonic_shared<kThreads>(s_who, e0 - s0);
                    for (uint32_t i = tid; i < e0 - s0; i += kThreads) s_order[s0 + i] = s_who[i];
                    __syncthreads();
                }
            }
            for (uint32_t q = tid; q < t; q += kThreads) a.ordenado[base + q] = s_order[q];
            // The bucket's records, gathered in order ("El kernel de
            // reordenación": destino[k] = origen[ordenado[k]]), through
            // stages in the cell table (warps 0-7) and the slot buffers
            // (warps 8-15), both free by now.  The copies write where the
            // threads wrote: order those writes first.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            {
                const uint32_t warp = tid >> 5;
                unsigned char *stage = reinterpret_cast<unsigned char *>(warp < kWarps / 2 ? s_table : s_who) +
                                       (size_t)(warp % (kWarps / 2)) * kStageBytes;
                gather_bucket(&origen_map, a, s_order, t, base, stage, smem_addr(&s_gbar[warp]), gather_uses,
                              &hdr->status);
            }
            __syncthreads();
            // The cell table, cleared for the next bucket.
#pragma unroll
            for (int q = 0; q < kScanVecs; ++q) s_held[q][tid] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (blockIdx.x == 0 && tid == 0) a.inicios[a.cells] = a.n;
    }
    if ((tid & 31u) == 0) bulk_wait_all();
    // The last CTA out: every bucket word has been zeroed.
    if (tid == 0 && atomicAdd(&hdr->bar_exit, 1u) == ctas - 1u) {
        if ((hdr->status & kStatusTimeout) == 0) hdr->buckets_clean = 1u;
        hdr->bar_count = 0u;
        hdr->bar_exit = 0u;
    }
}

std::atomic<int> g_grid[2][kMaxDevices];  // cached grid size per mode and device (0 = not yet known)

template <bool kStable>
cudaError_t bucketed_grid(int device, int *grid) {
    if (device >= 0 && device < kMaxDevices) {
        const int cached = g_grid[kStable][device].load(std::memory_order_relaxed);
        if (cached != 0) {
            *grid = cached;
            return cached > 0 ? cudaSuccess : cudaErrorNotSupported;
        }
    }
    int coop = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaFuncSetAttribute(build_bucketed_kernel<kStable>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDynamicSmem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_bucketed_kernel<kStable>, kThreads,
                                                          kDynamicSmem);
    if (e != cudaSuccess) return e;
    int gsz = coop ? per_sm * sms : -1;
    if (gsz <= 0 || gsz > (int)kFusedMaxCtas) gsz = -1;
    if (device >= 0 && device < kMaxDevices) g_grid[kStable][device].store(gsz, std::memory_order_relaxed);
    *grid = gsz;
    return gsz > 0 ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_build_bucketed(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                  uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                                  uint64_t cells, const Geometry &g, grid_ws_header *hdr, uint32_t *chunk_sums,
                                  uint32_t *slots, uint32_t *counts, uint32_t *total, uint32_t *base,
                                  uint32_t *pairs, bool stable, uint32_t *queue, uint32_t queue_capacity,
                                  uint32_t *sort_scratch, cudaStream_t s) {
    int device = 0, grid = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = stable ? bucketed_grid<true>(device, &grid) : bucketed_grid<false>(device, &grid);
    if (e != cudaSuccess) return e;
    const BucketPlan plan = bucket_plan(n, cells, (uint32_t)grid);
    if (plan.buckets == 0) return cudaErrorNotSupported;
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
    CUtensorMap map;
    if (record_tensor_map(origen, n, &map) != cudaSuccess) return cudaErrorNotSupported;
    const FusedScratch ws{chunk_sums, slots, counts, queue, queue_capacity, sort_scratch};
    const BucketScratch bk{plan.width, plan.buckets, plan.magic, total, base, reinterpret_cast<uint2 *>(pairs)};
    const BuildArgs a{reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino), conteos, celdaDe,
                      inicios, ordenado, n, cells};
    return cudaLaunchKernelEx(&cfg, stable ? build_bucketed_kernel<true> : build_bucketed_kernel<false>, map, a, g, hdr,
                              ws, bk);
}

}  // namespace ugrid
