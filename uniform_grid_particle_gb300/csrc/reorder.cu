// a5 — gather reorder of the 32-byte records into cell order.
//
// "Reordenar por celda y la coalescencia de memoria" (§El kernel de
// reordenación): destino[k] = origen[ordenado[k]].  A gather: the writes are
// contiguous and only the reads are scattered (the scatter direction is
// rejected on that page because scattered writes cost more).
//
// The records are fetched by the tensor memory accelerator: origen is a 2-D
// tensor of N rows of eight u32 words, and one tile::gather4 copy brings four
// whole rows, named by their indices, into shared memory.  Each warp owns a
// chunk of 128 output positions at a time: every lane reads four entries of
// ordenado and issues one gather4, an mbarrier counts the chunk's bytes in,
// and one bulk copy writes the 4 KB chunk to destino.  Two stages per warp
// keep a chunk in flight while the previous one is written.  No record passes
// through registers.  A chunk whose rows lie close together (an ordenado
// already near order) is read with 16-byte loads instead, which then share
// lines and sectors.
//
// A chunk holding an index >= N is not gathered either: the warp copies its
// valid records with plain loads and stores, skips the bad ones and sets the
// bounds status bit.
#include <algorithm>
#include <atomic>

#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kWarps = 8;
constexpr int kStages = 2;
constexpr uint32_t kChunk = 128;  // records per chunk: four per lane, one gather4 per lane
constexpr uint32_t kStageBytes = kChunk * sizeof(ugrid_particula);  // 4 KB
constexpr size_t kStageArea = (size_t)kWarps * kStages * kStageBytes;  // 64 KB
// After the stages: one mbarrier and one "plain loads" word per warp and stage.
constexpr size_t kSmemBytes = kStageArea + (size_t)kWarps * kStages * (sizeof(unsigned long long) + sizeof(uint32_t));
constexpr int kMaxDevices = 64;

__global__ void __launch_bounds__(32 * kWarps, 2)
reorder_kernel(const __grid_constant__ CUtensorMap origen_map, const uint32_t *__restrict__ ordenado,
               const uint4 *__restrict__ origen, uint4 *__restrict__ destino, uint32_t n, uint32_t *status) {
    extern __shared__ __align__(1024) unsigned char smem[];
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    unsigned char *stage = smem + (size_t)warp * kStages * kStageBytes;
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(smem + kStageArea) + warp * kStages;
    uint32_t *plain = reinterpret_cast<uint32_t *>(smem + kStageArea + (size_t)kWarps * kStages * 8) + warp * kStages;
    if ((smem_addr(smem) & 127u) != 0u) {  // the copies need 128-byte aligned stages
        if (threadIdx.x == 0) record_status(status, kStatusBounds);
        return;
    }
    if (lane < (uint32_t)kStages) mbar_init(smem_addr(bar + lane));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const uint32_t chunks = (uint32_t)(((uint64_t)n + kChunk - 1) / kChunk);
    const uint32_t first = blockIdx.x * kWarps + warp, stride = gridDim.x * kWarps;
    const uint32_t mine = first < chunks ? (chunks - 1u - first) / stride + 1u : 0u;

    // Chunk i of this warp into stage i % kStages.
    auto issue = [&](uint32_t i) {
        const uint32_t s = i % kStages;
        const uint64_t k0 = (uint64_t)(first + i * stride) * kChunk + 4u * lane;
        const uint32_t v = k0 < n ? (uint32_t)min((uint64_t)4, n - k0) : 0u;
        int row[4] = {0, 0, 0, 0};
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
        const uint32_t lanes = __popc(__ballot_sync(0xffffffffu, v > 0));
        if (lane_bad) record_status(status, kStatusBounds);
        // A chunk whose rows lie close together is read with 16-byte loads,
        // which then share lines and sectors, when it is written out.
        const bool near = !chunk_bad && rows_span(row, v) < kClusterRows;
        if (lane == 0) {
            plain[s] = chunk_bad || near ? 1u : 0u;
            mbar_arrive_expect(smem_addr(bar + s),
                               chunk_bad || near ? 0u : lanes * 4u * (uint32_t)sizeof(ugrid_particula));
        }
        __syncwarp();
        if (!chunk_bad && !near && v > 0)
            gather4_records(smem_addr(stage + s * kStageBytes + 4u * lane * sizeof(ugrid_particula)), &origen_map,
                            row, smem_addr(bar + s));
    };

    for (uint32_t i = 0; i < min(mine, (uint32_t)kStages); ++i) issue(i);
    for (uint32_t i = 0; i < mine; ++i) {
        const uint32_t s = i % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(bar + s), (i / kStages) & 1u))) {  // the warp agrees
            if (lane == 0) record_status(status, kStatusTimeout);
            // Let the other chunk in flight land (again with a limit) before
            // the CTA leaves.
            for (uint32_t j = i + 1; j < min(mine, i + kStages); ++j)
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(bar + j % kStages), (j / kStages) & 1u))) break;
            break;
        }
        const uint64_t k0 = (uint64_t)(first + i * stride) * kChunk;
        const uint32_t rows = (uint32_t)min((uint64_t)kChunk, n - k0);
        if (plain[s]) {
            // Rows close together, or one out of range: plain loads and
            // stores, four in flight per lane, skipping any bad row.
            for (uint32_t h0 = 0; h0 < 2u * rows; h0 += 4u * 32u) {
                uint32_t src[4];
                uint4 r4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t h = h0 + (uint32_t)k * 32u + lane;
                    src[k] = h < 2u * rows ? __ldg(ordenado + k0 + (h >> 1)) : n;
                    if (src[k] < n) r4[k] = load_nc_na(origen + 2 * (uint64_t)src[k] + (h & 1u));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (src[k] < n) store_cs(destino + 2 * k0 + h0 + (uint32_t)k * 32u + lane, r4[k]);
            }
        } else if (lane == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(destino + 2 * k0),
                         "r"(smem_addr(stage + s * kStageBytes)), "r"(rows * (uint32_t)sizeof(ugrid_particula))
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (i + kStages < mine) {
            // The stage is refilled only once its bulk copy has read it.
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
            issue(i + kStages);
        }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
    static std::atomic<EncodeTiled> fn{nullptr};
    EncodeTiled f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<EncodeTiled>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

std::atomic<int> g_ctas[kMaxDevices];  // grid size per device (0 = not yet known)

cudaError_t reorder_grid(int *ctas) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device >= 0 && device < kMaxDevices) {
        const int cached = g_ctas[device].load(std::memory_order_relaxed);
        if (cached > 0) {
            *ctas = cached;
            return cudaSuccess;
        }
    }
    int sms = 0, per_sm = 0;
    e = cudaFuncSetAttribute(reorder_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reorder_kernel, 32 * kWarps, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *ctas = sms * std::min(per_sm, 2);
    if (device >= 0 && device < kMaxDevices) g_ctas[device].store(*ctas, std::memory_order_relaxed);
    return cudaSuccess;
}

}  // namespace

cudaError_t rows_tensor_map(const void *base, uint32_t row_bytes, uint32_t rows, CUtensorMap *map) {
    if (row_bytes == 0 || row_bytes % 16 || row_bytes > 1024) return cudaErrorInvalidValue;
    const EncodeTiled encode = encode_tiled();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {row_bytes / 4, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {row_bytes / 4, 1};
    const cuuint32_t elem_strides[2] = {1, 1};
    if (encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box,
               elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t record_tensor_map(const ugrid_particula *origen, uint32_t n, CUtensorMap *map) {
    return rows_tensor_map(origen, (uint32_t)sizeof(ugrid_particula), n, map);
}

cudaError_t launch_reorder(const uint32_t *ordenado, const ugrid_particula *origen,
                           ugrid_particula *destino, uint32_t n, uint32_t *status, cudaStream_t s,
                           bool pdl) {
    if (n == 0) return cudaSuccess;
    CUtensorMap map;
    cudaError_t e = record_tensor_map(origen, n, &map);
    if (e != cudaSuccess) return e;
    int ctas = 0;
    e = reorder_grid(&ctas);
    if (e != cudaSuccess) return e;
    const uint64_t chunks = ((uint64_t)n + kChunk - 1) / kChunk;
    const unsigned grid = (unsigned)std::min<uint64_t>((uint64_t)ctas, (chunks + kWarps - 1) / kWarps);
    return launch(reorder_kernel, grid, 32 * kWarps, kSmemBytes, s, pdl, map, ordenado,
                  reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino), n, status);
}

}  // namespace ugrid
