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
#include "segsort_device.cuh"

namespace ugrid {
namespace {

constexpr int kSmallThreads = 256;
constexpr int kBigThreads = 512;
constexpr uint32_t kSharedMax = 16384;  // elements sorted in shared memory
constexpr size_t kBigSmemBytes = kSharedMax * sizeof(uint32_t);

static_assert(radix_smem_words<kBigThreads>() <= kSharedMax, "radix tier must fit in the shared buffer");

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
    if (!sort_short_segment(ordenado + a, b - a)) {
        const uint32_t q = atomicAdd(&hdr->stable_big, 1u);
        if (q < queue_capacity)
            queue[q] = (uint32_t)c;
        else
            record_status(&hdr->status, kStatusBounds);  // only inconsistent inicios get here
    }
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
        sort_long_segment<kBigThreads>(ordenado + a, scratch + a, len, n, smem, kSharedMax);
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
