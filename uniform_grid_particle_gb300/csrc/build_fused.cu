// The whole grid build in one cooperative launch.
//
// The pages chain separate dispatches because the phases depend on each other
// across workgroups ("Construir el índice de la rejilla…", §La cadena
// completa: the scan needs every count, the scatter every start).  Here every
// CTA of the grid is resident at once (cooperative launch, two CTAs per SM),
// so a grid-wide barrier stands in for each kernel boundary:
//
//   count   celdaDe[i] = cell of particle i; the atomic that counts it in the
//           workspace counter array returns its slot in the cell, kept in
//           slots[i]  ("Contar partículas por celda", §El kernel; the counter
//           array is also the cursor of "La dispersión").  Particles of one
//           CTA that share a cell are grouped first and take their slots with
//           one atomic (§La contención de las celdas densas)
//   scan a  each CTA totals one contiguous chunk of the counters
//   scan b  each CTA adds the totals of the chunks before it, scans its chunk
//           into inicios, copies the counts to conteos and zeroes its
//           counters; the last CTA writes inicios[C] = N
//                                                     ("Del conteo al inicio")
//   scatter ordenado[inicios[c] + slots[i]] = i        ("La dispersión")
//           and, in the same pass, destino[inicios[c] + slots[i]] = origen[i]
//
// The last line is the pages' gather destino[k] = origen[ordenado[k]] ("El
// kernel de reordenación") applied from the other side: the same permutation
// gives the same destino, and the phase, its barrier and the re-read of
// ordenado disappear.  Stable mode keeps a separate gather, because its
// places are known only once every cell's segment is sorted.
//
// Because the count's atomic already hands out the slot, the pages' second
// clear and second atomic pass are not needed: conteos ends as the histogram,
// exactly as after their cursor scatter, and every output is one the pages'
// chain can produce (order inside a cell is the atomics' arrival order).
//
// The counters live in the workspace and every build leaves them zero (scan b
// zeroes them after reading), so no clear phase is needed ("Poner a cero" is
// done by the previous build).  A header word records that they are clean; it
// is dropped while a build is using them, so a build that did not finish
// makes the next one clear them first.
//
// With GRID_STABLE two phases follow the scatter: one thread per cell sorts
// its segment in registers when it holds at most 32 particles and queues it
// otherwise, then CTAs take the queued segments one each (bitonic in shared
// memory up to 8192, an LSD radix sort through the workspace beyond).
//
// Particles (and the gather's half-records) are split into one contiguous,
// equal range per CTA, so every CTA has the same work in every phase.
//
// The count reads each record's first 16 bytes with an L2 evict-last policy
// and the record move (or the stable gather) reads the records with
// evict-first: the 32-byte sectors the count brings into L2 are still there
// when the records move.
//
// Grid barriers: a CTA arrives with a release add on a counter that only grows
// during the launch and waits, with acquire loads, until it reaches the number
// of CTAs times the barriers passed; the last CTA to leave the kernel resets
// it.  A wait gives up after kSpinLimitNs and records kStatusTimeout, so the
// kernel cannot hang (co-residency is guaranteed by the cooperative launch, so
// the limit is a guard, not part of the protocol).
#include <atomic>

#include "fused_common.cuh"

namespace ugrid {
namespace {

using namespace fused;

constexpr int kMaxDevices = 64;

template <bool kStable>
__global__ void __launch_bounds__(kThreads, 2)
build_fused_kernel(BuildArgs a, Geometry g, grid_ws_header *hdr, FusedScratch ws) {
    __shared__ uint32_t s_red[kWarps];
    __shared__ uint4 s_held[kScanVecs][kThreads];  // grouping table, then this CTA's chunk of counts (32 KB)
    __shared__ uint32_t s_clean;
    __shared__ uint32_t s_rows[kScanVecs + 1][kWarps];  // + the rows' totals
    const uint32_t tid = threadIdx.x;
    uint32_t passed = 0;  // grid barriers passed (thread 0)
    // Read before this CTA's first arrival, hence before anyone changes it.
    if (tid == 0) s_clean = *reinterpret_cast<volatile uint32_t *>(&hdr->counts_clean) >= a.cells;
    // Nobody touches the long-segment queue before the stable phases.
    if (kStable && blockIdx.x == 0 && tid == 0) hdr->stable_big = 0u;
    __syncthreads();
    uint64_t p_lo, p_hi;
    particle_range(a.n, p_lo, p_hi);

    // ---- clear the counters, only if the previous build did not leave them zero
    if (!s_clean) {
        clear_counters(ws.counts, a.cells);
        grid_barrier(hdr, passed);
    }

    count_phase<true>(a, g, ws, p_lo, p_hi, s_held);
    grid_barrier(hdr, passed);
    // The counters are not zero until the scan has run to the end.
    if (blockIdx.x == 0 && tid == 0) hdr->counts_clean = 0u;

    const ScanChunk chunk = scan_chunk(a.cells);
    scan_totals_phase(ws, chunk, s_held, s_red);
    grid_barrier(hdr, passed);

    scan_starts_phase(a, ws, chunk, s_held, s_red, s_rows);
    grid_barrier(hdr, passed);
    // Every CTA zeroed its counters before that barrier.
    if (blockIdx.x == 0 && tid == 0 && (hdr->status & kStatusTimeout) == 0)
        hdr->counts_clean = (uint32_t)a.cells;

    if constexpr (!kStable) {
        scatter_move_phase(a, ws, &hdr->status, p_lo, p_hi);
    } else {
        stable_tail_phase(a, ws, hdr, passed, p_lo, p_hi, s_held);
    }
    leave_launch(hdr);
}

std::atomic<int> g_grid[kMaxDevices];  // cached grid size per device (0 = not yet known)

cudaError_t fused_grid(int device, int *grid) {
    if (device >= 0 && device < kMaxDevices) {
        const int cached = g_grid[device].load(std::memory_order_relaxed);
        if (cached != 0) {
            *grid = cached;
            return cached > 0 ? cudaSuccess : cudaErrorNotSupported;
        }
    }
    int coop = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_fused_kernel<true>, kThreads, 0);
    if (e != cudaSuccess) return e;
    int g = coop ? per_sm * sms : -1;
    if (g == 0) g = -1;
    if (g > (int)kFusedMaxCtas) g = (int)kFusedMaxCtas;
    if (device >= 0 && device < kMaxDevices) g_grid[device].store(g, std::memory_order_relaxed);
    *grid = g;
    return g > 0 ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_build_fused(const ugrid_particula *origen, ugrid_particula *destino,
                               uint32_t *conteos, uint32_t *celdaDe, uint32_t *inicios,
                               uint32_t *ordenado, uint32_t n, uint64_t cells, const Geometry &g,
                               grid_ws_header *hdr, uint32_t *chunk_sums, uint32_t *slots,
                               uint32_t *counts, bool stable, uint32_t *queue,
                               uint32_t queue_capacity, uint32_t *sort_scratch, cudaStream_t s) {
    int device = 0, grid = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = fused_grid(device, &grid);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const FusedScratch ws{chunk_sums, slots, counts, queue, queue_capacity, sort_scratch};
    const BuildArgs a{reinterpret_cast<const uint4 *>(origen), reinterpret_cast<uint4 *>(destino), conteos, celdaDe,
                      inicios, ordenado, n, cells};
    return cudaLaunchKernelEx(&cfg, stable ? build_fused_kernel<true> : build_fused_kernel<false>, a, g, hdr, ws);
}

}  // namespace ugrid
