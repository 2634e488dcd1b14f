// a3 — exclusive scan of the per-cell counts, total in the extra slot.
//
// "Construir el índice de la rejilla con un prefix sum" (§Del conteo al
// inicio): inicios[c] = number of particles in the cells before c, and
// inicios[C] = N so that the end of cell c is inicios[c + 1].
//
// The pages use a three-level tree of 512-wide blocks (six dispatches).  Here
// it is one pass: tiles of 8192 cells, each CTA takes a tile ticket in arrival
// order, publishes its tile total, and finds its exclusive prefix by looking
// back over its predecessors' published words (decoupled look-back, Merrill &
// Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016).
//
// Look-back words are 64-bit: flag in the high half (0 = not yet published,
// 1 = tile total only, 2 = inclusive prefix), value in the low half, written
// and read with single relaxed gpu-scope accesses, `stride` words apart (in a
// workspace one per 128-byte line: every tile polls every earlier tile's
// word, and on a few dense lines those polls queued for microseconds).  One warp looks back over
// 256 predecessors per round (8 words per lane), so while all tiles of a
// 2M-cell grid are in flight a single round reaches tile 0; only that warp
// polls, and only the words closer than the nearest inclusive prefix are
// waited for.  Every wait gives up after kSpinLimitNs, records kStatusTimeout
// and carries on with a zero prefix, so a kernel never hangs.  Each CTA counts
// itself out once its look-back is done; the last one zeroes the words and
// the counters, leaving the workspace ready for the next call.
//
// Each tile is four rows of 2048 cells; thread t holds cells 4t..4t+3 of every
// row, so each row is read and written with fully coalesced 16-byte accesses.
//
// With zero_input (used by grid_build) each CTA also writes zeros over its
// tile of conteos after reading it: that is the second clear of the pages
// (the counter array reused as the scatter cursor), done with no extra pass.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr unsigned long long kFlagAggregate = 1ull << 32;
constexpr unsigned long long kFlagPrefix = 2ull << 32;
constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int kWarps = kScanThreads / 32;
constexpr int kRows = kScanItems / 4;
constexpr uint32_t kRowCells = kScanThreads * 4;
constexpr int kLookWords = 8;  // predecessors per lane per look-back round

__device__ __forceinline__ unsigned long long load_relaxed(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void store_relaxed(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t v) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFullMask, v, o);
        if (lane >= (uint32_t)o) v += t;
    }
    return v;
}

// Exclusive prefix of `tile` from its predecessors' words; called by one full
// warp.  Word w of lane l is predecessor j - (w*32 + l): the nearest one that
// shows an inclusive prefix ends the walk, and the tile totals of the closer
// ones are added to it.  Only the words closer than that prefix have to be
// published; pending ones are re-read together, one round trip per poll,
// with no sleep between polls (a sleep there cost microseconds).
__device__ uint32_t look_back(const unsigned long long *tile_status, uint32_t stride, uint32_t tile,
                              uint32_t *status_word) {
    const uint32_t lane = lane_id();
    uint32_t exclusive = 0;
    long long j = (long long)tile - 1;
    const unsigned long long start = global_ns();
    while (true) {
        unsigned long long s[kLookWords];
#pragma unroll
        for (int w = 0; w < kLookWords; ++w) {
            const long long idx = j - (long long)(w * 32 + lane);
            s[w] = idx >= 0 ? load_relaxed(tile_status + (uint64_t)idx * stride) : kFlagPrefix;
        }
        uint32_t nearest;
        while (true) {
            // Position (w*32 + lane) of the nearest inclusive prefix in the window.
            nearest = 0xffffffffu;
#pragma unroll
            for (int w = kLookWords - 1; w >= 0; --w)
                if ((s[w] >> 32) == 2) nearest = (uint32_t)(w * 32) + lane;
            nearest = __reduce_min_sync(kFullMask, nearest);
            bool pending = false;
#pragma unroll
            for (int w = 0; w < kLookWords; ++w)
                pending |= (uint32_t)(w * 32) + lane < nearest && (s[w] >> 32) == 0;
            if (!__any_sync(kFullMask, pending)) break;
            if (__shfl_sync(kFullMask, global_ns() - start > kSpinLimitNs, 0)) {
#pragma unroll
                for (int w = 0; w < kLookWords; ++w)
                    if ((s[w] >> 32) == 0) s[w] = kFlagPrefix;  // carry on with a zero prefix
                if (lane == 0) record_status(status_word, kStatusTimeout);
                continue;
            }
#pragma unroll
            for (int w = 0; w < kLookWords; ++w)
                if ((uint32_t)(w * 32) + lane < nearest && (s[w] >> 32) == 0)
                    s[w] = load_relaxed(tile_status + (uint64_t)(j - (long long)(w * 32 + lane)) * stride);
        }
        uint32_t sum = 0;
#pragma unroll
        for (int w = 0; w < kLookWords; ++w)
            if ((uint32_t)(w * 32) + lane <= nearest) sum += (uint32_t)s[w];
        exclusive += __reduce_add_sync(kFullMask, sum);
        if (nearest != 0xffffffffu) return exclusive;
        j -= 32 * kLookWords;
    }
}

// kZeroInput is the grid_build variant: it zeroes conteos after reading it,
// and it takes its tile ticket before waiting for the previous kernel (the
// count, which does not touch the workspace; the build's leading memset has
// already ordered it after any earlier scan on this workspace).
template <bool kZeroInput>
__global__ void __launch_bounds__(kScanThreads, 2)
scan_kernel(uint32_t *conteos, uint32_t *__restrict__ inicios, uint64_t cells, uint32_t tiles,
            grid_ws_header *hdr, unsigned long long *tile_status, uint32_t stride) {
    __shared__ uint32_t s_tile;
    __shared__ uint32_t s_warp[kRows][kWarps];
    __shared__ uint32_t s_row[kRows];
    __shared__ uint32_t s_prefix;
    __shared__ uint32_t s_last;
    const uint32_t tid = threadIdx.x;
    const uint32_t lane = tid & 31u;
    const uint32_t warp = tid >> 5;

    allow_dependent_launch();
    if (!kZeroInput) grid_dependency_wait();
    if (tid == 0) s_tile = atomicAdd(&hdr->scan_ticket, 1u);
    if (kZeroInput) grid_dependency_wait();
    __syncthreads();
    const uint32_t tile = s_tile;

    if (tile < tiles) {
        const uint64_t tile_base = (uint64_t)tile * kScanTile;
        uint4 v[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const uint64_t c = tile_base + (uint64_t)r * kRowCells + 4u * tid;
            if (c + 4 <= cells) {
                v[r] = *reinterpret_cast<const uint4 *>(conteos + c);
            } else {
                v[r].x = c + 0 < cells ? conteos[c + 0] : 0u;
                v[r].y = c + 1 < cells ? conteos[c + 1] : 0u;
                v[r].z = c + 2 < cells ? conteos[c + 2] : 0u;
                v[r].w = c + 3 < cells ? conteos[c + 3] : 0u;
            }
        }
        // Per row: the thread's total, its exclusive prefix inside the row.
        uint32_t total[kRows], excl[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            total[r] = v[r].x + v[r].y + v[r].z + v[r].w;
            const uint32_t incl = warp_inclusive_sum(total[r]);
            excl[r] = incl - total[r];
            if (lane == 31) s_warp[r][warp] = incl;
        }
        __syncthreads();
        if (warp < kRows) {  // warp r scans the warp totals of row r
            const uint32_t w = lane < kWarps ? s_warp[warp][lane] : 0u;
            const uint32_t wi = warp_inclusive_sum(w);
            if (lane < kWarps) s_warp[warp][lane] = wi - w;
            if (lane == kWarps - 1) s_row[warp] = wi;
        }
        __syncthreads();
        uint32_t row_off[kRows];
        uint32_t tile_total = 0;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            row_off[r] = tile_total;
            tile_total += s_row[r];
        }

        // Publish the tile total, then find the prefix of all earlier tiles.
        if (warp == 0) {
            uint32_t exclusive = 0;
            if (tile == 0) {
                if (lane == 0) store_relaxed(tile_status, kFlagPrefix | tile_total);
            } else {
                if (lane == 0) store_relaxed(tile_status + (uint64_t)tile * stride, kFlagAggregate | tile_total);
                exclusive = look_back(tile_status, stride, tile, &hdr->status);
                if (lane == 0)
                    store_relaxed(tile_status + (uint64_t)tile * stride,
                                  kFlagPrefix | (uint32_t)(exclusive + tile_total));
            }
            if (lane == 0) s_prefix = exclusive;
        }
        __syncthreads();
        // This CTA reads no more look-back words: count it out now, so the
        // last one can clear them while the others still write inicios.  The
        // fence orders this CTA's last publish (by this same thread) before
        // the count-out, so the last CTA's reset cannot be overtaken by it.
        if (tid == 0) {
            __threadfence();
            s_last = atomicAdd(&hdr->scan_done, 1u) == gridDim.x - 1 ? 1u : 0u;
        }

        const uint32_t prefix = s_prefix;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const uint64_t c = tile_base + (uint64_t)r * kRowCells + 4u * tid;
            uint4 o;
            o.x = prefix + row_off[r] + s_warp[r][warp] + excl[r];
            o.y = o.x + v[r].x;
            o.z = o.y + v[r].y;
            o.w = o.z + v[r].z;
            if (c + 4 <= cells) {
                *reinterpret_cast<uint4 *>(inicios + c) = o;
                if (kZeroInput) *reinterpret_cast<uint4 *>(conteos + c) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                const uint32_t ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (c + k < cells) {
                        inicios[c + k] = ov[k];
                        if (kZeroInput) conteos[c + k] = 0u;
                    }
                }
            }
        }
        if (tile == tiles - 1 && tid == 0) inicios[cells] = prefix + tile_total;
    } else if (tid == 0) {
        record_status(&hdr->status, kStatusBounds);  // more CTAs than tiles: a stale ticket
        __threadfence();
        s_last = atomicAdd(&hdr->scan_done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }

    // The last CTA counted out resets the look-back words and the counters.
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (uint32_t t = tid; t < tiles; t += kScanThreads) tile_status[(uint64_t)t * stride] = 0ull;
        if (tid == 0) {
            hdr->scan_ticket = 0u;
            hdr->scan_done = 0u;
        }
    }
}

}  // namespace

cudaError_t launch_scan(uint32_t *conteos, uint32_t *inicios, uint64_t cells, bool zero_input,
                        grid_ws_header *hdr, unsigned long long *tile_status, uint32_t stride, cudaStream_t s,
                        bool pdl) {
    const uint32_t tiles = (uint32_t)scan_tiles(cells);
    if (zero_input)
        return launch(scan_kernel<true>, tiles, kScanThreads, 0, s, pdl, conteos, inicios, cells,
                      tiles, hdr, tile_status, stride);
    return launch(scan_kernel<false>, tiles, kScanThreads, 0, s, pdl, conteos, inicios, cells,
                  tiles, hdr, tile_status, stride);
}

}  // namespace ugrid
