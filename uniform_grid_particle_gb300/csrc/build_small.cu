// The whole grid build for a small scene, in one CTA and one launch.
//
// A scene of at most kSmallMaxParticles particles on at most kSmallMaxCells
// cells fits one CTA's shared memory whole: the cell table, each particle's
// cell and slot, and the cell order.  One CTA then runs the pages' chain
// with no grid-wide dependency to cross ("Construir el índice de la rejilla
// con un prefix sum", §La cadena completa: the phases are separate dispatches
// only because their dependencies span the whole grid):
//   count   celdaDe[i] = cell of particle i ("Contar partículas por celda",
//           §El kernel); the slot it takes in its cell's shared counter
//   scan    conteos and inicios = the counts and their exclusive scan, with
//           inicios[C] = N (§Del conteo al inicio)
//   place   ordenado[inicios[c] + slot] = i (§La dispersión), in shared memory;
//           in stable mode every cell's segment then sorted by particle index
//           (§El orden dentro de la celda)
//   gather  destino[k] = origen[ordenado[k]] ("Reordenar por celda…", §El
//           kernel de reordenación)
// The multi-CTA builds pay two grid barriers and a prologue per CTA for
// scenes like this; here the whole build is a few shared-memory passes.
#include <atomic>

#include "ugrid_internal.cuh"
#include "segsort_device.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kCellsPerThread = kSmallMaxCells / kThreads;  // 8: two 16-byte vectors
static_assert(kCellsPerThread == 8, "each thread scans two vectors of four cells");
constexpr uint32_t kItems = kSmallMaxParticles / kThreads;  // particles per thread
constexpr uint32_t kSlotBits = 13;                          // slot < kSmallMaxParticles
static_assert((1u << kSlotBits) == kSmallMaxParticles && (1u << kSlotBits) == kSmallMaxCells,
              "a cell and a slot pack into one word");
constexpr uint32_t kLongMax = kSmallMaxParticles / (kRegisterMax + 1) + 1;
constexpr size_t kDynamicSmem = 3 * (size_t)kSmallMaxCells * sizeof(uint32_t);  // table, place, order

template <bool kStable>
__global__ void __launch_bounds__(kThreads, 1)
build_small_kernel(const uint4 *__restrict__ origen, uint4 *__restrict__ destino, uint32_t *__restrict__ conteos,
                   uint32_t *__restrict__ celdaDe, uint32_t *__restrict__ inicios, uint32_t *__restrict__ ordenado,
                   uint32_t n, uint32_t cells, Geometry g) {
    extern __shared__ __align__(16) uint32_t s_dyn[];
    uint32_t *s_table = s_dyn;                        // [kSmallMaxCells] counts, then starts
    uint32_t *s_place = s_table + kSmallMaxCells;     // [kSmallMaxParticles] cell << kSlotBits | slot
    uint32_t *s_order = s_place + kSmallMaxParticles; // [kSmallMaxParticles] the cell order
    __shared__ uint32_t s_warp[2][kWarps];
    __shared__ uint32_t s_long[kLongMax];
    __shared__ uint32_t s_nlong;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;

    reinterpret_cast<uint4 *>(s_table)[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(s_table)[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) s_nlong = 0u;
    __syncthreads();

    // count: the records' positions (16-byte loads), cells, slots
    {
        uint4 rec[kItems];
#pragma unroll
        for (uint32_t k = 0; k < kItems; ++k) {
            const uint32_t i = k * kThreads + tid;
            if (i < n) rec[k] = load_nc_na(origen + 2 * (uint64_t)i);
        }
#pragma unroll
        for (uint32_t k = 0; k < kItems; ++k) {
            const uint32_t i = k * kThreads + tid;
            const bool valid = i < n;
            const uint32_t c = valid ? cell_of(rec[k], g) : 0u;
            const uint32_t slot = smem_take(s_table, valid, c);
            if (valid) {
                celdaDe[i] = c;
                s_place[i] = c << kSlotBits | slot;
            }
        }
    }
    __syncthreads();

    // scan: thread t holds cells 8t .. 8t+7
    {
        const uint4 v0 = reinterpret_cast<const uint4 *>(s_table)[2 * tid];
        const uint4 v1 = reinterpret_cast<const uint4 *>(s_table)[2 * tid + 1];
        const uint32_t c8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t total = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) total += c8[e];
        uint32_t incl = total;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t up = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= (uint32_t)o) incl += up;
        }
        if (lane == 31) s_warp[0][warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint32_t wt = s_warp[0][lane];
            uint32_t wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t up = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= (uint32_t)o) wi += up;
            }
            s_warp[1][lane] = wi - wt;
        }
        __syncthreads();
        uint32_t start = s_warp[1][warp] + incl - total;
        uint32_t st[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            st[e] = start;
            start += c8[e];
        }
        const uint32_t c0 = 8u * tid;
        if (c0 + 8 <= cells) {
            reinterpret_cast<uint4 *>(conteos + c0)[0] = v0;
            reinterpret_cast<uint4 *>(conteos + c0)[1] = v1;
            reinterpret_cast<uint4 *>(inicios + c0)[0] = make_uint4(st[0], st[1], st[2], st[3]);
            reinterpret_cast<uint4 *>(inicios + c0)[1] = make_uint4(st[4], st[5], st[6], st[7]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (c0 + e < cells) {
                    conteos[c0 + e] = c8[e];
                    inicios[c0 + e] = st[e];
                }
            }
        }
        if (tid == 0) inicios[cells] = n;
        reinterpret_cast<uint4 *>(s_table)[2 * tid] = make_uint4(st[0], st[1], st[2], st[3]);
        reinterpret_cast<uint4 *>(s_table)[2 * tid + 1] = make_uint4(st[4], st[5], st[6], st[7]);
    }
    __syncthreads();

    // place
    for (uint32_t i = tid; i < n; i += kThreads) {
        const uint32_t p = s_place[i];
        s_order[s_table[p >> kSlotBits] + (p & ((1u << kSlotBits) - 1u))] = i;
    }
    __syncthreads();

    if constexpr (kStable) {
        // Every cell's segment sorted by particle index: short ones by one
        // thread in registers, longer ones by the whole CTA in shared memory
        // (s_place is free by now).
        for (uint32_t c = tid; c < cells; c += kThreads) {
            const uint32_t s0 = s_table[c], e0 = c + 1 < cells ? s_table[c + 1] : n;
            if (e0 > s0 + 1 && !sort_short_segment(s_order + s0, e0 - s0)) {
                const uint32_t q = atomicAdd(&s_nlong, 1u);
                if (q < kLongMax) s_long[q] = c;
            }
        }
        __syncthreads();
        const uint32_t nlong = min(s_nlong, kLongMax);
        for (uint32_t q = 0; q < nlong; ++q) {
            const uint32_t c = s_long[q];
            const uint32_t s0 = s_table[c], e0 = c + 1 < cells ? s_table[c + 1] : n;
            for (uint32_t i = tid; i < e0 - s0; i += kThreads) s_place[i] = s_order[s0 + i];
            bitonic_shared<kThreads>(s_place, e0 - s0);
            for (uint32_t i = tid; i < e0 - s0; i += kThreads) s_order[s0 + i] = s_place[i];
            __syncthreads();
        }
    }

    // ordenado, then the records in cell order: two threads per record, every
    // half-record load of a round issued before its stores
    for (uint32_t k = tid; k < n; k += kThreads) ordenado[k] = s_order[k];
    constexpr uint32_t kHalves = 4;
    for (uint32_t h0 = 0; h0 < 2u * n; h0 += kHalves * kThreads) {
        uint4 v[kHalves];
#pragma unroll
        for (uint32_t e = 0; e < kHalves; ++e) {
            const uint32_t h = h0 + e * kThreads + tid;
            if (h < 2u * n) v[e] = load_nc_na(origen + 2 * (uint64_t)s_order[h >> 1] + (h & 1u));
        }
#pragma unroll
        for (uint32_t e = 0; e < kHalves; ++e) {
            const uint32_t h = h0 + e * kThreads + tid;
            if (h < 2u * n) store_cs(destino + h, v[e]);
        }
    }
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_configured[2][kMaxDevices];  // per mode and device: shared-memory size set

}  // namespace

cudaError_t launch_build_small(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                               uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n,
                               uint32_t cells, const Geometry &g, bool stable, cudaStream_t s) {
    auto kernel = stable ? build_small_kernel<true> : build_small_kernel<false>;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const bool cacheable = device >= 0 && device < kMaxDevices;
    if (!cacheable || !g_configured[stable][device].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynamicSmem);
        if (e != cudaSuccess) return e;
        if (cacheable) g_configured[stable][device].store(true, std::memory_order_release);
    }
    return launch(kernel, 1u, kThreads, kDynamicSmem, s, false, reinterpret_cast<const uint4 *>(origen),
                  reinterpret_cast<uint4 *>(destino), conteos, celdaDe, inicios, ordenado, n, cells, g);
}

}  // namespace ugrid
