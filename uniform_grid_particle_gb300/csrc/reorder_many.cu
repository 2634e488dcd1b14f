// Gather reorder of several particle arrays with one index read.
//
// "Reordenar por celda y la coalescencia de memoria" (§El kernel de
// reordenación): when the particle state lives in several buffers — the hot
// Cinematica and the cold Aspecto of "El estado de las partículas en storage
// buffers" (§AoS o SoA) — the same ordenado is applied to all of them, and one
// kernel that reads ordenado[k] once for every pair is better than one kernel
// per pair.  For every array a and every k < N:
//     destino_a[k] = origen_a[ordenado[k]]   (records of record_bytes_a bytes)
//
// Arrays of records of at most 64 bytes are fetched by the tensor memory
// accelerator, as in the single-array reorder: each array is a 2-D tensor of N
// rows, and a warp takes chunks of 128 consecutive positions k, one array at a
// time.  Every lane reads ordenado[k0 + 4l .. k0 + 4l + 3] and issues one
// tile::gather4 copy of those four rows into its own slot of the warp's stage
// (a 128-byte aligned slot of 128 or 256 bytes: a copy's shared-memory
// destination must be 128-byte aligned, and four 16- or 48-byte rows do not
// fill one), an mbarrier counts the chunk in, and the warp writes the stage out
// with coalesced 16-byte stores.  Two stages per warp keep one (chunk, array)
// in flight while the previous one is written.  A chunk whose rows lie close
// together, or that holds an index >= N, is copied with plain 16-byte loads
// (the bad records skipped, status bit set).
//
// Larger records take the plain kernel: each warp takes chunks of 128
// consecutive positions k: lane l reads ordenado[k0 + 32e + l] for e = 0..3
// (four coalesced 128-byte reads), then, for every array and every 16-byte
// piece of a record, loads the piece of each of its four records before any
// store, and stores them so that one store instruction of the warp writes the
// pieces of 32 consecutive positions.  A position whose index is >= N is
// skipped (status bit set).
#include <algorithm>
#include <atomic>

#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerCta = kThreads / 32;
constexpr uint32_t kChunk = 128;    // positions per warp chunk, four per lane
constexpr uint32_t kInFlight = 8;   // 16-byte pieces a lane loads before it stores

__global__ void __launch_bounds__(kThreads)
reorder_many_kernel(const uint32_t *__restrict__ ordenado, const __grid_constant__ ManyArrays m, uint32_t n,
                    uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t chunks = (uint32_t)(((uint64_t)n + kChunk - 1) / kChunk);
    const uint32_t stride = gridDim.x * kWarpsPerCta;
    for (uint32_t c = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); c < chunks; c += stride) {
        const uint64_t k0 = (uint64_t)c * kChunk;
        uint32_t src[4];
        bool ok[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint64_t k = k0 + 32u * e + lane;
            src[e] = k < n ? __ldg(ordenado + k) : n;
            ok[e] = src[e] < n;
            if (k < n && !ok[e]) record_status(status, kStatusBounds);
        }
        // Pieces in order (array a, piece p, position e), kInFlight at a time.
        const uint32_t total = 4u * m.per_record;
        for (uint32_t g0 = 0; g0 < total; g0 += kInFlight) {
            uint4 v[kInFlight];
#pragma unroll
            for (uint32_t i = 0; i < kInFlight; ++i) {
                const uint32_t gi = g0 + i;
                if (gi < total) {
                    const uint32_t piece = gi >> 2, e = gi & 3u;
                    uint32_t a = 0;
                    while (a + 1 < m.count && piece >= m.first[a + 1]) ++a;
                    const uint32_t pp = piece - m.first[a];
                    if (ok[e]) v[i] = load_nc_na(m.src[a] + (uint64_t)src[e] * m.pieces[a] + pp);
                }
            }
#pragma unroll
            for (uint32_t i = 0; i < kInFlight; ++i) {
                const uint32_t gi = g0 + i;
                if (gi < total) {
                    const uint32_t piece = gi >> 2, e = gi & 3u;
                    uint32_t a = 0;
                    while (a + 1 < m.count && piece >= m.first[a + 1]) ++a;
                    const uint32_t pp = piece - m.first[a];
                    const uint64_t k = k0 + 32u * e + lane;
                    if (ok[e]) store_cs(m.dst[a] + k * m.pieces[a] + pp, v[i]);
                }
            }
        }
    }
}

// ---- the tensor-memory-accelerator form, records of at most 64 bytes ----------

constexpr int kTmaWarps = 8;
constexpr int kTmaStages = 2;
constexpr uint32_t kTmaMaxRecord = 64;  // four rows fill at most a 256-byte slot

struct ManyMaps {
    CUtensorMap map[kMaxArrays];  // array a as N rows of bytes[a] bytes
    uint4 *dst[kMaxArrays];
    const uint4 *src[kMaxArrays];
    uint32_t bytes[kMaxArrays];   // record bytes of each array
    uint32_t count;               // arrays in use
    uint32_t slot;                // bytes of a lane's slot: four records of the widest array, 128-byte aligned
};

constexpr size_t tma_smem_bytes(uint32_t slot) {
    return (size_t)kTmaWarps * kTmaStages * 32u * slot +
           (size_t)kTmaWarps * kTmaStages * (sizeof(unsigned long long) + sizeof(uint32_t));
}

// The record position of 16-byte piece h when a record has `pieces` pieces
// (1 to 4 in the TMA form): a shift or a multiply, not a division.
__device__ __forceinline__ uint32_t position_of(uint32_t h, uint32_t pieces) {
    switch (pieces) {
        case 1: return h;
        case 2: return h >> 1;
        case 3: return h / 3u;
        default: return h >> 2;
    }
}

__global__ void __launch_bounds__(32 * kTmaWarps)
reorder_many_tma_kernel(const __grid_constant__ ManyMaps m, const uint32_t *__restrict__ ordenado, uint32_t n,
                        uint32_t *status) {
    extern __shared__ __align__(1024) unsigned char smem[];
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t stage_bytes = 32u * m.slot;
    const size_t area = (size_t)kTmaWarps * kTmaStages * stage_bytes;
    unsigned char *stage = smem + (size_t)warp * kTmaStages * stage_bytes;
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(smem + area) + warp * kTmaStages;
    uint32_t *plain = reinterpret_cast<uint32_t *>(smem + area + (size_t)kTmaWarps * kTmaStages * 8) + warp * kTmaStages;
    if ((smem_addr(smem) & 127u) != 0u) {  // the copies need 128-byte aligned slots
        if (threadIdx.x == 0) record_status(status, kStatusBounds);
        return;
    }
    if (lane < (uint32_t)kTmaStages) mbar_init(smem_addr(bar + lane));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const uint32_t chunks = (uint32_t)(((uint64_t)n + kChunk - 1) / kChunk);
    const uint32_t first = blockIdx.x * kTmaWarps + warp, stride = gridDim.x * kTmaWarps;
    const uint32_t mine = first < chunks ? (chunks - 1u - first) / stride + 1u : 0u;
    const uint32_t items = mine * m.count;  // item i: this warp's chunk i / count, array i % count

    // The item to issue next, and the lane's rows of its chunk: the arrays of
    // one chunk are issued one after another and share the rows.
    uint32_t iss_chunk = 0, iss_array = 0;
    int row[4] = {0, 0, 0, 0};
    uint32_t v = 0, lanes = 0;
    bool copy_plain = true;
    auto issue = [&](uint32_t i) {
        const uint32_t s = i % kTmaStages, a = iss_array;
        const uint64_t k0 = (uint64_t)(first + iss_chunk * stride) * kChunk + 4u * lane;
        if (a == 0) {
            v = k0 < n ? (uint32_t)min((uint64_t)4, n - k0) : 0u;
            bool lane_bad = false;
            if (v > 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t r = __ldg(ordenado + k0 + min((uint32_t)e, v - 1u));
                    lane_bad |= r >= n;
                    row[e] = (int)r;
                }
            }
            const bool chunk_bad = __any_sync(0xffffffffu, lane_bad);
            lanes = __popc(__ballot_sync(0xffffffffu, v > 0));
            if (lane_bad) record_status(status, kStatusBounds);
            copy_plain = chunk_bad || rows_span(row, v) < kClusterRows;
        }
        if (lane == 0) {
            plain[s] = copy_plain ? 1u : 0u;
            mbar_arrive_expect(smem_addr(bar + s), copy_plain ? 0u : lanes * 4u * m.bytes[a]);
        }
        __syncwarp();
        if (!copy_plain && v > 0)
            gather4_records(smem_addr(stage + s * stage_bytes + lane * m.slot), &m.map[a], row, smem_addr(bar + s));
        if (++iss_array == m.count) {
            iss_array = 0;
            ++iss_chunk;
        }
    };

    for (uint32_t i = 0; i < min(items, (uint32_t)kTmaStages); ++i) issue(i);
    uint32_t chunk = 0, a = 0;  // the item being written out
    for (uint32_t i = 0; i < items; ++i) {
        const uint32_t s = i % kTmaStages;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(bar + s), (i / kTmaStages) & 1u))) {  // the warp agrees
            if (lane == 0) record_status(status, kStatusTimeout);
            for (uint32_t j = i + 1; j < min(items, i + kTmaStages); ++j)
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(bar + j % kTmaStages), (j / kTmaStages) & 1u))) break;
            break;
        }
        const uint64_t k0 = (uint64_t)(first + chunk * stride) * kChunk;
        const uint32_t rows = (uint32_t)min((uint64_t)kChunk, n - k0);
        const uint32_t pieces = m.bytes[a] / 16u, total = rows * pieces;
        uint4 *dst = m.dst[a] + k0 * pieces;
        if (plain[s]) {
            // Rows close together, or one out of range: 16-byte loads, four
            // in flight per lane, skipping any bad row.
            const uint4 *src = m.src[a];
            for (uint32_t h0 = 0; h0 < total; h0 += 4u * 32u) {
                uint32_t from[4];
                uint4 r4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t h = h0 + (uint32_t)k * 32u + lane;
                    const uint32_t p = position_of(h, pieces);
                    from[k] = h < total ? __ldg(ordenado + k0 + p) : n;
                    if (from[k] < n) r4[k] = load_nc_na(src + (uint64_t)from[k] * pieces + (h - p * pieces));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (from[k] < n) store_cs(dst + h0 + (uint32_t)k * 32u + lane, r4[k]);
            }
        } else {
            // Position p sits in lane p / 4's slot, row p % 4: one 16-byte
            // piece per lane and store, 32 consecutive pieces per warp store.
            const unsigned char *st = stage + s * stage_bytes;
            for (uint32_t h = lane; h < total; h += 32u) {
                const uint32_t p = position_of(h, pieces);
                const uint4 val = *reinterpret_cast<const uint4 *>(st + (p >> 2) * m.slot + (p & 3u) * m.bytes[a] +
                                                                   (h - p * pieces) * 16u);
                store_cs(dst + h, val);
            }
        }
        if (i + kTmaStages < items) {
            // Every lane has read the stage before any lane's copy refills it.
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(i + kTmaStages);
        }
        if (++a == m.count) {
            a = 0;
            ++chunk;
        }
    }
    __syncwarp();
}

std::atomic<int> g_ctas[64];         // grid size per device (0 = not yet known)
std::atomic<int> g_tma_ctas[64][2];  // the same for the TMA form, 128- and 256-byte slots

// CTAs of the TMA form on this device for slots of `slot` bytes (128 or 256).
// The kernel's shared-memory limit is raised once to what 256-byte slots need,
// so calls with either slot size can run side by side.
cudaError_t tma_grid(uint32_t slot, int *ctas) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const int which = slot > 128u ? 1 : 0;
    const bool cache = device >= 0 && device < 64;
    if (cache) {
        const int cached = g_tma_ctas[device][which].load(std::memory_order_relaxed);
        if (cached > 0) {
            *ctas = cached;
            return cudaSuccess;
        }
    }
    int sms = 0, per_sm = 0;
    e = cudaFuncSetAttribute(reorder_many_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tma_smem_bytes(2u * 128u));
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reorder_many_tma_kernel, 32 * kTmaWarps,
                                                          tma_smem_bytes(slot));
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *ctas = sms * std::min(per_sm, 2);
    if (cache) g_tma_ctas[device][which].store(*ctas, std::memory_order_relaxed);
    return cudaSuccess;
}

// The TMA form for these arrays, or cudaErrorNotSupported when a record is
// wider than 64 bytes or a tensor map cannot be made.
cudaError_t launch_many_tma(const uint32_t *ordenado, const ManyArrays &arrays, uint32_t n, uint32_t *status,
                            cudaStream_t s, bool pdl) {
    if (n > 0x7fffffffu) return cudaErrorNotSupported;  // row coordinates are signed 32-bit
    ManyMaps m{};
    m.count = arrays.count;
    m.slot = 128u;
    for (uint32_t a = 0; a < arrays.count; ++a) {
        const uint32_t bytes = arrays.pieces[a] * 16u;
        if (bytes > kTmaMaxRecord) return cudaErrorNotSupported;
        if (rows_tensor_map(arrays.src[a], bytes, n, &m.map[a]) != cudaSuccess) return cudaErrorNotSupported;
        m.src[a] = arrays.src[a];
        m.dst[a] = arrays.dst[a];
        m.bytes[a] = bytes;
        m.slot = std::max(m.slot, (4u * bytes + 127u) & ~127u);
    }
    int ctas = 0;
    cudaError_t e = tma_grid(m.slot, &ctas);
    if (e != cudaSuccess) return e;
    const uint64_t chunks = ((uint64_t)n + kChunk - 1) / kChunk;
    const unsigned grid = (unsigned)std::min<uint64_t>((uint64_t)ctas, (chunks + kTmaWarps - 1) / kTmaWarps);
    return launch(reorder_many_tma_kernel, grid, 32 * kTmaWarps, tma_smem_bytes(m.slot), s, pdl, m, ordenado, n,
                  status);
}

}  // namespace

cudaError_t launch_reorder_many(const uint32_t *ordenado, const ManyArrays &m, uint32_t n,
                                uint32_t *status, cudaStream_t s, bool pdl) {
    if (n == 0) return cudaSuccess;
    {
        const cudaError_t t = launch_many_tma(ordenado, m, n, status, s, pdl);
        if (t != cudaErrorNotSupported) return t;
    }
    int device = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    int ctas = device >= 0 && device < 64 ? g_ctas[device].load(std::memory_order_relaxed) : 0;
    if (ctas == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reorder_many_kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        ctas = std::max(1, sms * per_sm);
        if (device >= 0 && device < 64) g_ctas[device].store(ctas, std::memory_order_relaxed);
    }
    const uint64_t chunks = ((uint64_t)n + kChunk - 1) / kChunk;
    const unsigned grid =
        (unsigned)std::min<uint64_t>((uint64_t)ctas, (chunks + kWarpsPerCta - 1) / kWarpsPerCta);
    return launch(reorder_many_kernel, grid, kThreads, 0, s, pdl, ordenado, m, n, status);
}

}  // namespace ugrid
