// a3 — exclusive scan of the per-cell counts, total in the extra slot.
//
// "Construir el índice de la rejilla con un prefix sum" (§Del conteo al
// inicio): inicios[c] = number of particles in the cells before c, and
// inicios[C] = N so that the end of cell c is inicios[c + 1].
//
// The pages use a three-level tree of 512-wide blocks (six dispatches).  Here
// it is one pass: tiles of 4096 cells, each CTA takes a tile ticket in arrival
// order, publishes its tile total, and finds its exclusive prefix by looking
// back over its predecessors' published words (decoupled look-back, Merrill &
// Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016).
//
// Look-back words are 64-bit: flag in the high half (0 = not yet published,
// 1 = tile total only, 2 = inclusive prefix), value in the low half, written
// and read with single relaxed gpu-scope accesses.  Every wait gives up after
// kSpinLimitNs, records kStatusTimeout and carries on with a zero prefix, so
// a kernel never hangs.  The last CTA to finish zeroes the words and the
// counters, leaving the workspace ready for the next call.
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

// Exclusive prefix of `tile` from its predecessors' words; called by one
// full warp.  Lane l inspects tile j - l, 32 tiles per round, until some
// predecessor shows an inclusive prefix.
__device__ uint32_t look_back(const unsigned long long *tile_status, uint32_t tile,
                              uint32_t *status_word) {
    const uint32_t lane = lane_id();
    uint32_t exclusive = 0;
    long long j = (long long)tile - 1;
    unsigned long long start = 0;
    while (true) {
        const long long idx = j - (long long)lane;
        unsigned long long s = idx >= 0 ? load_relaxed(tile_status + idx) : kFlagPrefix;
        while (__any_sync(kFullMask, (s >> 32) == 0)) {
            if (start == 0) start = global_ns();
            const bool give_up = __shfl_sync(kFullMask, (global_ns() - start) > kSpinLimitNs, 0);
            if (give_up) {
                if ((s >> 32) == 0) s = kFlagPrefix;  // carry on with a zero prefix
                if (lane == 0) record_status(status_word, kStatusTimeout);
                break;
            }
            __nanosleep(32);
            if ((s >> 32) == 0) s = load_relaxed(tile_status + idx);
        }
        const uint32_t prefix_lanes = __ballot_sync(kFullMask, (s >> 32) == 2);
        uint32_t value = (uint32_t)s;
        if (prefix_lanes) {
            const uint32_t stop = (uint32_t)(__ffs(prefix_lanes) - 1);
            if (lane > stop) value = 0;
            return exclusive + __reduce_add_sync(kFullMask, value);
        }
        exclusive += __reduce_add_sync(kFullMask, value);
        j -= 32;
    }
}

template <bool kZeroInput>
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(uint32_t *conteos, uint32_t *__restrict__ inicios, uint64_t cells, uint32_t tiles,
            grid_ws_header *hdr, unsigned long long *tile_status) {
    __shared__ uint32_t s_tile;
    __shared__ uint32_t s_warp[kWarps];
    __shared__ uint32_t s_total;
    __shared__ uint32_t s_prefix;
    __shared__ uint32_t s_last;
    const uint32_t tid = threadIdx.x;
    const uint32_t lane = tid & 31u;
    const uint32_t warp = tid >> 5;

    if (tid == 0) s_tile = atomicAdd(&hdr->scan_ticket, 1u);
    __syncthreads();
    const uint32_t tile = s_tile;

    if (tile < tiles) {
        const uint64_t base = (uint64_t)tile * kScanTile + (uint64_t)tid * kScanItems;
        const bool full = base + kScanItems <= cells;
        uint32_t v[kScanItems];
        if (full) {
            const uint4 *src = reinterpret_cast<const uint4 *>(conteos + base);
#pragma unroll
            for (int q = 0; q < kScanItems / 4; ++q) {
                const uint4 x = src[q];
                v[4 * q + 0] = x.x;
                v[4 * q + 1] = x.y;
                v[4 * q + 2] = x.z;
                v[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < kScanItems; ++k) v[k] = base + k < cells ? conteos[base + k] : 0u;
        }
        // Thread-local exclusive scan; `run` is the thread's total.
        uint32_t run = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const uint32_t t = v[k];
            v[k] = run;
            run += t;
        }
        // Block-wide exclusive scan of the thread totals.
        const uint32_t incl = warp_inclusive_sum(run);
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint32_t w = lane < kWarps ? s_warp[lane] : 0u;
            const uint32_t wi = warp_inclusive_sum(w);
            if (lane < kWarps) s_warp[lane] = wi - w;
            if (lane == kWarps - 1) s_total = wi;
        }
        __syncthreads();
        const uint32_t thread_excl = s_warp[warp] + incl - run;

        // Publish the tile total, then find the prefix of all earlier tiles.
        if (warp == 0) {
            const uint32_t total = s_total;
            uint32_t exclusive = 0;
            if (tile == 0) {
                if (lane == 0) store_relaxed(tile_status, kFlagPrefix | total);
            } else {
                if (lane == 0) store_relaxed(tile_status + tile, kFlagAggregate | total);
                exclusive = look_back(tile_status, tile, &hdr->status);
                if (lane == 0) store_relaxed(tile_status + tile, kFlagPrefix | (uint32_t)(exclusive + total));
            }
            if (lane == 0) s_prefix = exclusive;
        }
        __syncthreads();

        const uint32_t prefix = s_prefix + thread_excl;
        if (full) {
            uint4 *dst = reinterpret_cast<uint4 *>(inicios + base);
#pragma unroll
            for (int q = 0; q < kScanItems / 4; ++q)
                dst[q] = make_uint4(prefix + v[4 * q], prefix + v[4 * q + 1], prefix + v[4 * q + 2],
                                    prefix + v[4 * q + 3]);
            if (kZeroInput) {
                uint4 *z = reinterpret_cast<uint4 *>(conteos + base);
#pragma unroll
                for (int q = 0; q < kScanItems / 4; ++q) z[q] = make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < kScanItems; ++k) {
                if (base + k < cells) {
                    inicios[base + k] = prefix + v[k];
                    if (kZeroInput) conteos[base + k] = 0u;
                }
            }
        }
        if (tile == tiles - 1 && tid == 0) inicios[cells] = s_prefix + s_total;
    } else if (tid == 0) {
        record_status(&hdr->status, kStatusBounds);  // more CTAs than tiles: a stale ticket
    }

    // The last CTA out resets the look-back words and the counters.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&hdr->scan_done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (uint32_t t = tid; t < tiles; t += kScanThreads) tile_status[t] = 0ull;
        if (tid == 0) {
            hdr->scan_ticket = 0u;
            hdr->scan_done = 0u;
        }
    }
}

}  // namespace

cudaError_t launch_scan(uint32_t *conteos, uint32_t *inicios, uint64_t cells, bool zero_input,
                        grid_ws_header *hdr, unsigned long long *tile_status, cudaStream_t s) {
    const uint32_t tiles = (uint32_t)scan_tiles(cells);
    if (zero_input)
        scan_kernel<true><<<tiles, kScanThreads, 0, s>>>(conteos, inicios, cells, tiles, hdr, tile_status);
    else
        scan_kernel<false><<<tiles, kScanThreads, 0, s>>>(conteos, inicios, cells, tiles, hdr, tile_status);
    return cudaGetLastError();
}

}  // namespace ugrid
