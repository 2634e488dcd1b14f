// a6 — stable mode: every cell's segment of ordenado sorted by particle index.
//
// "Construir el índice de la rejilla con un prefix sum" (§El orden dentro de
// la celda): the atomic cursor hands out slots in arrival order, so two runs
// group the particles the same way but order each cell differently.  The
// page's middle way is a second pass that sorts each cell using the particle
// index as the tie-break, with a small network when cells hold a few dozen
// particles.  Sorting every segment ascending gives exactly the stable
// counting-sort order.
//
// Tiers by segment length L:
//   L <= 1           nothing to do;
//   2 <= L <= 32     one thread, a bitonic network over registers (8/16/32);
//   32 < L <= 16384  queued; one CTA sorts it in shared memory (bitonic);
//   L > 16384        queued; one CTA runs an LSD radix sort (8-bit digits)
//                    through the workspace scratch, stably ranking each
//                    chunk with __match_any_sync and per-warp digit counts.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kSmallThreads = 256;
constexpr int kRegisterMax = 32;
constexpr int kBigThreads = 512;
constexpr int kBigWarps = kBigThreads / 32;
constexpr uint32_t kSharedMax = 16384;  // elements sorted in shared memory
constexpr size_t kBigSmemBytes = kSharedMax * sizeof(uint32_t);
constexpr uint32_t kPad = 0xffffffffu;

static_assert((256 + 256 + kBigWarps * 256) * sizeof(uint32_t) <= kBigSmemBytes,
              "radix tier must fit in the shared buffer");

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
    for (int k = 0; k < M; ++k) r[k] = (uint32_t)k < len ? seg[k] : kPad;
    bitonic_registers<M>(r);
#pragma unroll
    for (int k = 0; k < M; ++k)
        if ((uint32_t)k < len) seg[k] = r[k];
}

// One thread per cell: short segments sorted in place, long ones queued.
__global__ void __launch_bounds__(kSmallThreads)
segment_small_kernel(const uint32_t *__restrict__ inicios, uint32_t *__restrict__ ordenado,
                     uint32_t n, uint32_t cells, grid_ws_header *hdr, uint32_t *queue,
                     uint32_t queue_capacity) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t c = (uint64_t)blockIdx.x * kSmallThreads + threadIdx.x;
    if (c >= cells) return;
    const uint32_t a = inicios[c];
    const uint32_t b = inicios[c + 1];
    if (b < a || b > n) {
        record_status(&hdr->status, kStatusBounds);
        return;
    }
    const uint32_t len = b - a;
    if (len <= 1) return;
    uint32_t *seg = ordenado + a;
    if (len <= 8)
        sort_in_registers<8>(seg, len);
    else if (len <= 16)
        sort_in_registers<16>(seg, len);
    else if (len <= kRegisterMax)
        sort_in_registers<kRegisterMax>(seg, len);
    else {
        const uint32_t q = atomicAdd(&hdr->stable_big, 1u);
        if (q < queue_capacity)
            queue[q] = (uint32_t)c;
        else
            record_status(&hdr->status, kStatusBounds);  // only inconsistent inicios get here
    }
}

__device__ void bitonic_shared(uint32_t *buf, uint32_t len) {
    uint32_t p = 1;
    while (p < len) p <<= 1;
    for (uint32_t i = len + threadIdx.x; i < p; i += kBigThreads) buf[i] = kPad;
    __syncthreads();
    for (uint32_t k = 2; k <= p; k <<= 1) {
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t i = threadIdx.x; i < p; i += kBigThreads) {
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

// Stable LSD radix sort of seg[0..len) (values < n), ping-ponging with tmp.
__device__ void radix_global(uint32_t *seg, uint32_t *tmp, uint32_t len, uint32_t n,
                             uint32_t *smem) {
    uint32_t *hist = smem;              // [256] digit totals, then running offsets
    uint32_t *scan = smem + 256;        // [256] scratch for the offset scan
    uint32_t *wc = smem + 512;          // [kBigWarps][256] per-warp digit counts
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t bits = 32u - __clz(n - 1u);
    const uint32_t passes = (bits + 7u) / 8u;
    uint32_t *src = seg, *dst = tmp;
    for (uint32_t pass = 0; pass < passes; ++pass) {
        const uint32_t shift = 8u * pass;
        for (uint32_t d = tid; d < 256; d += kBigThreads) hist[d] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < len; i += kBigThreads) atomicAdd(&hist[(src[i] >> shift) & 255u], 1u);
        __syncthreads();
        if (tid == 0) {  // 256 entries: a serial scan is cheap next to the passes
            uint32_t run = 0;
            for (int d = 0; d < 256; ++d) {
                scan[d] = run;
                run += hist[d];
            }
        }
        __syncthreads();
        for (uint32_t d = tid; d < 256; d += kBigThreads) hist[d] = scan[d];
        __syncthreads();
        for (uint32_t base = 0; base < len; base += kBigThreads) {
            const uint32_t idx = base + tid;
            const bool valid = idx < len;
            const uint32_t v = valid ? src[idx] : 0u;
            const uint32_t d = (v >> shift) & 255u;
            for (uint32_t e = tid; e < kBigWarps * 256; e += kBigThreads) wc[e] = 0;
            __syncthreads();
            const uint32_t active = __ballot_sync(0xffffffffu, valid);
            uint32_t rank = 0;
            if (valid) {
                const uint32_t peers = __match_any_sync(active, d);
                rank = __popc(peers & lanemask_lt());
                if (lane == (uint32_t)(__ffs(peers) - 1)) wc[warp * 256 + d] = __popc(peers);
            }
            __syncthreads();
            for (uint32_t dd = tid; dd < 256; dd += kBigThreads) {
                uint32_t run = hist[dd];
                for (int w = 0; w < kBigWarps; ++w) {
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
        for (uint32_t i = tid; i < len; i += kBigThreads) seg[i] = src[i];
    }
    __syncthreads();
}

// Persistent CTAs work through the queue of long segments.
__global__ void __launch_bounds__(kBigThreads)
segment_big_kernel(const uint32_t *__restrict__ inicios, uint32_t *__restrict__ ordenado,
                   uint32_t n, grid_ws_header *hdr, const uint32_t *__restrict__ queue,
                   uint32_t queue_capacity, uint32_t *scratch) {
    extern __shared__ uint32_t smem[];
    __shared__ uint32_t s_last;
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t queued = *(volatile uint32_t *)&hdr->stable_big;
    const uint32_t count = queued < queue_capacity ? queued : queue_capacity;
    for (uint32_t q = blockIdx.x; q < count; q += gridDim.x) {
        const uint32_t c = queue[q];
        const uint32_t a = inicios[c];
        const uint32_t len = inicios[c + 1] - a;
        if (len <= kSharedMax) {
            for (uint32_t i = threadIdx.x; i < len; i += kBigThreads) smem[i] = ordenado[a + i];
            bitonic_shared(smem, len);
            for (uint32_t i = threadIdx.x; i < len; i += kBigThreads) ordenado[a + i] = smem[i];
            __syncthreads();
        } else {
            radix_global(ordenado + a, scratch + a, len, n, smem);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&hdr->stable_done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
        hdr->stable_big = 0u;
        hdr->stable_done = 0u;
    }
}

}  // namespace

size_t segment_queue_capacity(uint64_t n, uint64_t cells) {
    const uint64_t longest = n / (kRegisterMax + 1) + 1;  // cells longer than 32
    return (size_t)(longest < cells ? longest : cells);
}

cudaError_t launch_segment_sort(const uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                                uint32_t cells, grid_ws_header *hdr, uint32_t *queue,
                                uint32_t *scratch, cudaStream_t s, bool pdl) {
    if (n < 2) return cudaSuccess;
    const uint32_t capacity = (uint32_t)segment_queue_capacity(n, cells);
    const unsigned small_blocks = (unsigned)((cells + kSmallThreads - 1) / kSmallThreads);
    cudaError_t e = launch(segment_small_kernel, small_blocks, kSmallThreads, 0, s, pdl, inicios,
                           ordenado, n, cells, hdr, queue, capacity);
    if (e != cudaSuccess) return e;
    int device = 0, sms = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(segment_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kBigSmemBytes)) != cudaSuccess)
        return e;
    return launch(segment_big_kernel, (unsigned)sms, kBigThreads, kBigSmemBytes, s, pdl, inicios,
                  ordenado, n, hdr, queue, capacity, scratch);
}

}  // namespace ugrid
