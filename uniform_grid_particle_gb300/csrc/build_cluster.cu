// The grid build for small scenes on one thread-block cluster: the CTAs of the
// cluster share one cell table in distributed shared memory.
//
// A scene of at most kClusterMaxParticles particles on at most
// kClusterMaxCells cells needs no grid-wide step: the cluster's CTAs (one per
// SM) each own a slice of the cells' counters in their shared memory and
// reach the others' slices directly.  The pages' chain ("Construir el índice
// de la rejilla con un prefix sum", §La cadena completa) then runs as:
//   count    celdaDe[i] = cell of particle i ("Contar partículas por celda",
//            §El kernel), and the particle's slot = an atomic add on its
//            cell's counter in the owning CTA's slice
//   scan     each CTA scans its slice; the slices' totals are exchanged, so
//            every CTA knows where its cells start: conteos and inicios
//            (§Del conteo al inicio, inicios[C] = N)
//   scatter  ordenado[inicios[c] + slot] = i (§La dispersión), the start read
//            from the owning CTA's slice, and the record copied to
//            destino[inicios[c] + slot] by the same thread: every record is
//            read once in order and written once, so no gather pass is
//            needed ("Reordenar por celda…", §El kernel de reordenación:
//            destino[k] = origen[ordenado[k]] holds by construction)
// The order within a cell is that of the atomics, so the cluster build serves the
// non-stable mode; stable builds of small scenes take the one-CTA build.
#include <atomic>

#include <cooperative_groups.h>

#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 1024;
constexpr uint32_t kItems = kClusterMaxParticles / (kClusterMaxCtas * kThreads);  // particles per thread
constexpr uint32_t kSliceMax = kClusterMaxCells / kClusterMaxCtas;  // cells per CTA's slice, at most
constexpr uint32_t kCellsPerThread = kSliceMax / kThreads;         // 8: two 16-byte vectors
static_assert(kCellsPerThread == 8, "each thread scans two vectors of four cells");
static_assert(kItems * kClusterMaxCtas * kThreads == kClusterMaxParticles, "whole rounds of particles");
constexpr int kWarps = kThreads / 32;

// Cluster-wide slot take on the counter of `cell` (in CTA `owner`'s slice at
// `local`): a plain remote atomic per lane, unless some lane's cell equals the
// cell of the lane below it, then one atomic per distinct cell of the warp.
// Every lane of the warp must call it.
__device__ __forceinline__ uint32_t cluster_take(cg::cluster_group &cluster, uint32_t *s_count, bool valid,
                                                 uint32_t cell, uint32_t owner, uint32_t local) {
    uint32_t *counter = valid ? cluster.map_shared_rank(s_count, (int)owner) + local : nullptr;
    if (!warp_has_adjacent_duplicates(valid, cell)) return valid ? atomicAdd(counter, 1u) : 0u;
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    if (!valid) return 0u;
    const uint32_t peers = __match_any_sync(active, cell);
    const uint32_t leader = (uint32_t)(__ffs(peers) - 1);
    uint32_t first = 0u;
    if (lane_id() == leader) first = atomicAdd(counter, (uint32_t)__popc(peers));
    first = __shfl_sync(peers, first, leader);
    return first + (uint32_t)__popc(peers & lanemask_lt());
}

__global__ void __launch_bounds__(kThreads, 1)
build_cluster_kernel(const uint4 *__restrict__ origen, uint4 *__restrict__ destino, uint32_t *__restrict__ conteos,
                     uint32_t *__restrict__ celdaDe, uint32_t *__restrict__ inicios, uint32_t *__restrict__ ordenado,
                     uint32_t n, uint32_t cells, uint32_t slice, Geometry g) {
    __shared__ __align__(16) uint32_t s_count[kSliceMax];  // this CTA's cells: counts, then first positions
    __shared__ uint32_t s_total[kClusterMaxCtas];          // every CTA's particle total
    __shared__ uint32_t s_warp[2][kWarps];
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t rank = cluster.block_rank(), ctas = cluster.num_blocks();
    reinterpret_cast<uint4 *>(s_count)[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(s_count)[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
    // Every slice zeroed before any remote add; the barrier completes while
    // the records load (split: arrive now, wait before the adds).
    cluster.barrier_arrive();

    // count: this CTA's particles [p0, p1)
    const uint32_t p0 = (uint32_t)((uint64_t)n * rank / ctas), p1 = (uint32_t)((uint64_t)n * (rank + 1) / ctas);
    uint4 head[kItems];
    uint32_t cell[kItems], slot[kItems];
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        if (i < p1) head[k] = load_nc_na(origen + 2 * (uint64_t)i);
    }
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        cell[k] = i < p1 ? cell_of(head[k], g) : 0u;  // celdaDe written at the end
    }
    cluster.barrier_wait();
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        const uint32_t owner = cell[k] / slice;
        slot[k] = cluster_take(cluster, s_count, i < p1, cell[k], owner, cell[k] - owner * slice);
    }
    cluster.sync();  // every count in

    // scan: thread t holds cells 8t .. 8t+7 of the slice
    {
        const uint4 v0 = reinterpret_cast<const uint4 *>(s_count)[2 * tid];
        const uint4 v1 = reinterpret_cast<const uint4 *>(s_count)[2 * tid + 1];
        const uint32_t c8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += c8[e];
        uint32_t incl = sum;
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
            // this slice's total to every CTA of the cluster
            if (lane == 31)
                for (uint32_t r = 0; r < ctas; ++r) *cluster.map_shared_rank(&s_total[rank], (int)r) = wi;
        }
        cluster.sync();  // every slice total in (and s_warp[1] for this CTA)
        uint32_t before = 0;
        for (uint32_t r = 0; r < rank; ++r) before += s_total[r];
        uint32_t start = before + s_warp[1][warp] + incl - sum;
        uint32_t st[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            st[e] = start;
            start += c8[e];
        }
        reinterpret_cast<uint4 *>(s_count)[2 * tid] = make_uint4(st[0], st[1], st[2], st[3]);
        reinterpret_cast<uint4 *>(s_count)[2 * tid + 1] = make_uint4(st[4], st[5], st[6], st[7]);
        // Every slice's starts in place: the arrival releases them; conteos
        // and inicios are stored while the barrier completes (a release
        // waits for the stores before it, so they come after).
        cluster.barrier_arrive();
        const uint32_t lo = rank * slice, hi = min(cells, lo + slice);  // this slice's cells
        const uint32_t c0 = lo + 8u * tid;
        if (8u * tid < slice && c0 + 8 <= hi) {
            reinterpret_cast<uint4 *>(conteos + c0)[0] = v0;
            reinterpret_cast<uint4 *>(conteos + c0)[1] = v1;
            reinterpret_cast<uint4 *>(inicios + c0)[0] = make_uint4(st[0], st[1], st[2], st[3]);
            reinterpret_cast<uint4 *>(inicios + c0)[1] = make_uint4(st[4], st[5], st[6], st[7]);
        } else if (8u * tid < slice) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (8u * tid + e < slice && c0 + e < hi) {
                    conteos[c0 + e] = c8[e];
                    inicios[c0 + e] = st[e];
                }
            }
        }
        if (rank == ctas - 1 && tid == 0) inicios[cells] = n;
    }
    cluster.barrier_wait();

    // scatter: each particle to its position, with its record.  The starts
    // are read from the owners' slices first; the closing barrier (no CTA
    // leaves while another may still read its slice) completes during the
    // stores.
    uint32_t pos[kItems];
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        if (i < p1) {
            const uint32_t owner = cell[k] / slice;
            pos[k] = *(cluster.map_shared_rank(s_count, (int)owner) + (cell[k] - owner * slice)) + slot[k];
        }
    }
    // The arrival releases: the remote loads above are performed before it
    // (the records' second halves are loaded after it, so that it does not
    // wait for them too).
    cluster.barrier_arrive();
    uint4 tail[kItems];
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        if (i < p1) tail[k] = load_nc_na(origen + 2 * (uint64_t)i + 1);
    }
#pragma unroll
    for (uint32_t k = 0; k < kItems; ++k) {
        const uint32_t i = p0 + k * kThreads + tid;
        if (i < p1) {
            celdaDe[i] = cell[k];
            ordenado[pos[k]] = i;
            store_cs(destino + 2 * (uint64_t)pos[k], head[k]);
            store_cs(destino + 2 * (uint64_t)pos[k] + 1, tail[k]);
        }
    }
    cluster.barrier_wait();
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_ctas[kMaxDevices];  // per device: cluster size that launches (0 = not yet known, -1 = none)

// The largest cluster of kClusterMaxCtas or fewer (a power of two, at least
// 8) that the device can run.
int cluster_ctas(int device) {
    const bool cacheable = device >= 0 && device < kMaxDevices;
    if (cacheable) {
        const int cached = g_ctas[device].load(std::memory_order_relaxed);
        if (cached != 0) return cached;
    }
    int found = -1;
    if (cudaFuncSetAttribute(build_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        for (int k = (int)kClusterMaxCtas; k >= 8 && found < 0; k /= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)k);
            cfg.blockDim = dim3(kThreads);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)k;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, build_cluster_kernel, &cfg) == cudaSuccess && clusters > 0)
                found = k;
        }
    }
    (void)cudaGetLastError();
    if (cacheable) g_ctas[device].store(found, std::memory_order_relaxed);
    return found;
}

}  // namespace

cudaError_t launch_build_cluster(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
                                 uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, uint32_t n, uint32_t cells,
                                 const Geometry &g, cudaStream_t s) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const int k = cluster_ctas(device);
    if (k <= 0 || n == 0 || n > (uint32_t)k * kItems * kThreads || (uint64_t)cells > (uint64_t)k * kSliceMax)
        return cudaErrorNotSupported;
    // Slices of whole 16-byte vectors, so that every slice starts aligned.
    uint32_t slice = (cells + (uint32_t)k - 1) / (uint32_t)k;
    slice = (slice + 3u) & ~3u;
    if (slice > kSliceMax) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)k);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, build_cluster_kernel, reinterpret_cast<const uint4 *>(origen),
                              reinterpret_cast<uint4 *>(destino), conteos, celdaDe, inicios, ordenado, n, cells, slice,
                              g);
}

}  // namespace ugrid
