// Device routines of the stable mode's segment sort, shared by the segment-sort
// kernels and the single-launch builds (fused and bucketed).
//
// "Construir el índice de la rejilla con un prefix sum" (§El orden dentro de
// la celda): sorting every cell's segment of ordenado by particle index gives
// the stable counting-sort order; for cells of a few dozen particles a small
// network does it cheaply.
#pragma once

#include "ugrid_internal.cuh"

namespace ugrid {

constexpr int kRegisterMax = 32;  // longest segment sorted by one thread in registers
constexpr uint32_t kSortPad = 0xffffffffu;

template <int M>
__device__ __forceinline__ void bitonic_registers(uint32_t (&r)[M]) {
#pragma unroll
    for (int k = 2; k <= M; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const uint32_t a = r[i], b = r[l];
                    const bool ascending = (i & k) == 0;
                    r[i] = ascending ? min(a, b) : max(a, b);
                    r[l] = ascending ? max(a, b) : min(a, b);
                }
            }
        }
    }
}

template <int M>
__device__ __forceinline__ void sort_in_registers(uint32_t *seg, uint32_t len) {
    uint32_t r[M];
#pragma unroll
    for (int k = 0; k < M; ++k) r[k] = (uint32_t)k < len ? seg[k] : kSortPad;
    bitonic_registers<M>(r);
#pragma unroll
    for (int k = 0; k < M; ++k)
        if ((uint32_t)k < len) seg[k] = r[k];
}

__device__ __forceinline__ void compare_exchange(uint32_t &a, uint32_t &b) {
    const uint32_t lo = min(a, b), hi = max(a, b);
    a = lo;
    b = hi;
}

// Sorts seg[0..len) in the calling thread when len <= kRegisterMax; returns
// false (nothing done) for longer segments.  Two to four elements, the common
// lengths at a few particles per cell, take their optimal networks (1, 3 and
// 5 compare-exchanges); longer ones a bitonic network of 8, 16 or 32.
__device__ __forceinline__ bool sort_short_segment(uint32_t *seg, uint32_t len) {
    if (len <= 1) return true;
    if (len <= 4) {
        uint32_t a = seg[0], b = seg[1];
        if (len == 2) {
            if (a > b) {
                seg[0] = b;
                seg[1] = a;
            }
            return true;
        }
        uint32_t c = seg[2];
        if (len == 3) {
            compare_exchange(a, b);
            compare_exchange(b, c);
            compare_exchange(a, b);
            seg[0] = a;
            seg[1] = b;
            seg[2] = c;
            return true;
        }
        uint32_t d = seg[3];
        compare_exchange(a, b);
        compare_exchange(c, d);
        compare_exchange(a, c);
        compare_exchange(b, d);
        compare_exchange(b, c);
        seg[0] = a;
        seg[1] = b;
        seg[2] = c;
        seg[3] = d;
        return true;
    }
    if (len <= 8)
        sort_in_registers<8>(seg, len);
    else if (len <= 16)
        sort_in_registers<16>(seg, len);
    else if (len <= kRegisterMax)
        sort_in_registers<kRegisterMax>(seg, len);
    else
        return false;
    return true;
}

// Bitonic sort of buf[0..len) in shared memory by a whole CTA of THREADS
// threads; buf must hold the next power of two >= len.
template <int THREADS>
__device__ void bitonic_shared(uint32_t *buf, uint32_t len) {
    uint32_t p = 1;
    while (p < len) p <<= 1;
    for (uint32_t i = len + threadIdx.x; i < p; i += THREADS) buf[i] = kSortPad;
    __syncthreads();
    for (uint32_t k = 2; k <= p; k <<= 1) {
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t i = threadIdx.x; i < p; i += THREADS) {
                const uint32_t l = i ^ j;
                if (l > i) {
                    const uint32_t a = buf[i], b = buf[l];
                    const bool ascending = (i & k) == 0;
                    if ((a > b) == ascending) {
                        buf[i] = b;
                        buf[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Shared-memory words radix_global needs for a CTA of THREADS threads.
template <int THREADS>
constexpr uint32_t radix_smem_words() {
    return 512u + (uint32_t)(THREADS / 32) * 256u;
}

// Stable LSD radix sort (8-bit digits) of seg[0..len), values < n, by a whole
// CTA of THREADS threads, ping-ponging with tmp[0..len).  Each chunk of
// THREADS values is ranked stably: __match_any_sync gives a value's rank among
// the lower lanes of its warp with the same digit, and per-warp digit counts,
// turned into running offsets in warp order, place the warps one after the
// other.  smem must hold radix_smem_words<THREADS>() words.
template <int THREADS>
__device__ void radix_global(uint32_t *seg, uint32_t *tmp, uint32_t len, uint32_t n, uint32_t *smem) {
    constexpr int kWarpsPerCta = THREADS / 32;
    uint32_t *hist = smem;        // [256] digit totals, then running offsets
    uint32_t *scan = smem + 256;  // [256] scratch for the offset scan
    uint32_t *wc = smem + 512;    // [warps][256] per-warp digit counts
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t bits = 32u - __clz(n - 1u);
    const uint32_t passes = (bits + 7u) / 8u;
    uint32_t *src = seg, *dst = tmp;
    for (uint32_t pass = 0; pass < passes; ++pass) {
        const uint32_t shift = 8u * pass;
        for (uint32_t d = tid; d < 256; d += THREADS) hist[d] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < len; i += THREADS) atomicAdd(&hist[(src[i] >> shift) & 255u], 1u);
        __syncthreads();
        if (tid == 0) {  // 256 entries: a serial scan is cheap next to the passes
            uint32_t run = 0;
            for (int d = 0; d < 256; ++d) {
                scan[d] = run;
                run += hist[d];
            }
        }
        __syncthreads();
        for (uint32_t d = tid; d < 256; d += THREADS) hist[d] = scan[d];
        __syncthreads();
        for (uint32_t base = 0; base < len; base += THREADS) {
            const uint32_t idx = base + tid;
            const bool valid = idx < len;
            const uint32_t v = valid ? src[idx] : 0u;
            const uint32_t d = (v >> shift) & 255u;
            for (uint32_t e = tid; e < kWarpsPerCta * 256u; e += THREADS) wc[e] = 0;
            __syncthreads();
            const uint32_t active = __ballot_sync(0xffffffffu, valid);
            uint32_t rank = 0;
            if (valid) {
                const uint32_t peers = __match_any_sync(active, d);
                rank = __popc(peers & lanemask_lt());
                if (lane == (uint32_t)(__ffs(peers) - 1)) wc[warp * 256 + d] = __popc(peers);
            }
            __syncthreads();
            for (uint32_t dd = tid; dd < 256; dd += THREADS) {
                uint32_t run = hist[dd];
                for (int w = 0; w < kWarpsPerCta; ++w) {
                    const uint32_t t = wc[w * 256 + dd];
                    wc[w * 256 + dd] = run;
                    run += t;
                }
                hist[dd] = run;
            }
            __syncthreads();
            if (valid) dst[wc[warp * 256 + d] + rank] = v;
            __syncthreads();
        }
        uint32_t *t = src;
        src = dst;
        dst = t;
    }
    if (src != seg) {
        for (uint32_t i = tid; i < len; i += THREADS) seg[i] = src[i];
    }
    __syncthreads();
}

// Sorts one long segment seg[0..len) with a whole CTA: in shared memory
// (bitonic) when it fits in `smem_words` (a power of two, at least
// radix_smem_words<THREADS>()), otherwise by radix through `tmp`.  The bitonic
// path needs the next power of two >= len words of smem.
template <int THREADS>
__device__ void sort_long_segment(uint32_t *seg, uint32_t *tmp, uint32_t len, uint32_t n,
                                  uint32_t *smem, uint32_t smem_words) {
    uint32_t padded = 1;  // the bitonic sort fills up to the next power of two
    while (padded < len) padded <<= 1;
    if (padded <= smem_words) {
        for (uint32_t i = threadIdx.x; i < len; i += THREADS) smem[i] = seg[i];
        bitonic_shared<THREADS>(smem, len);
        for (uint32_t i = threadIdx.x; i < len; i += THREADS) seg[i] = smem[i];
        __syncthreads();
    } else {
        radix_global<THREADS>(seg, tmp, len, n, smem);
    }
}

}  // namespace ugrid
