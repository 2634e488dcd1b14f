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
// Each warp takes chunks of 128 consecutive positions k: lane l reads
// ordenado[k0 + 32e + l] for e = 0..3 (four coalesced 128-byte reads), then,
// for every array and every 16-byte piece of a record, loads the piece of each
// of its four records before any store, and stores them so that one store
// instruction of the warp writes the pieces of 32 consecutive positions.  A
// position whose index is >= N is skipped (status bit set).
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

std::atomic<int> g_ctas[64];  // grid size per device (0 = not yet known)

}  // namespace

cudaError_t launch_reorder_many(const uint32_t *ordenado, const ManyArrays &m, uint32_t n,
                                uint32_t *status, cudaStream_t s, bool pdl) {
    if (n == 0) return cudaSuccess;
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
