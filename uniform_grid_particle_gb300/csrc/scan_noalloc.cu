// grid_scan_noalloc: the exclusive scan of grid_scan with its scratch held in
// a fixed array inside the library, so the caller passes only its input and
// output.
//
// Who needs it: some callers may not take device memory of their own when
// they want a scan.  An engine or framework that owns every device buffer and
// hands them out from its own pool, or a per-frame simulation step that must
// not risk cudaMalloc (which can synchronise the device and take unbounded
// time), cannot provide the workspace grid_scan asks for.  For them the
// library keeps the few kilobytes the scan needs in a static device array.
//
// The scratch: a 256-byte header (the status word, the tile-ticket and
// finished-tile counters) followed by one 64-bit look-back word per 8192-cell
// tile, for at most kNoAllocMaxTiles tiles: 33,024 bytes, which every device
// that loads the library holds until the process exits.  Inputs of more than
// kNoAllocMaxCells cells are rejected with GRID_ERANGE before any CUDA call.
//
// Host code never uses the array's name as a device address (in host code it
// names a host-side stand-in).  The first call on each device, with that device
// current, looks the address up with cudaGetSymbolAddress and caches it with
// the device's current context; make that first call before capturing any
// stream.  A call that finds another context current (the primary context
// was reset and created again, so the module and its array were loaded
// anew) looks the address up again.  Every call clears the header
// and the look-back words it will use with cudaMemsetAsync on its stream, then
// launches the same scan kernel as grid_scan.  All calls share the one array:
// calls whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on it and must be serialised by the caller.
// Device-side diagnostics (a look-back wait that gave up) land in the array's
// status word and are not reported by this entry point.
#include <cmath>
#include <mutex>

#include "ugrid_internal.cuh"

namespace {

constexpr uint64_t kNoAllocMaxTiles = 4096;
constexpr uint64_t kNoAllocMaxCells = kNoAllocMaxTiles * ugrid::kScanTile;  // 33,554,432
constexpr size_t kNoAllocScratchBytes =
    ugrid::kHeaderBytes + kNoAllocMaxTiles * sizeof(unsigned long long);

static __device__ __align__(256) unsigned char g_scan_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The array's address on each device, and the context it was looked up in.
struct CachedAddress {
    CUcontext ctx;
    void *ptr;
};
CachedAddress g_scratch_address[kMaxDevices];
std::mutex g_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// cuCtxGetCurrent from the driver, looked up through the runtime once.
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// Device address of g_scan_scratch on the current device, looked up once per
// device and context and cached.  Before the runtime has made the device's
// context current the driver reports none; the symbol lookup then creates it.
cudaError_t scratch_address(void **out) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const CtxGetCurrentFn get = ctx_get_current();
    if (get == nullptr) return cudaErrorDeviceUninitialized;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    const bool cacheable = device >= 0 && device < kMaxDevices;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (cacheable && ctx != nullptr && g_scratch_address[device].ctx == ctx) {
        *out = g_scratch_address[device].ptr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    if (cacheable) g_scratch_address[device] = CachedAddress{ctx, p};
    *out = p;
    return cudaSuccess;
}

bool params_ok(const grid_params *p) {
    if (p == nullptr) return false;
    uint64_t c = 1;
    for (int d = 0; d < 3; ++d) {
        if (p->dims[d] == 0) return false;
        c *= p->dims[d];
        if (c > 0xfffffffeull) return false;
    }
    if (c != p->celdas) return false;
    for (int d = 0; d < 3; ++d)
        if (!std::isfinite(p->origin[d])) return false;
    return std::isfinite(p->cellSize) && p->cellSize > 0.0f && std::isfinite(1.0f / p->cellSize);
}

}  // namespace

extern "C" int grid_scan_noalloc(const uint32_t *conteos, uint32_t *inicios, const grid_params *p,
                                 void *stream) {
    if (!params_ok(p)) return GRID_EINVAL;
    const uint64_t cells = p->celdas;
    if (cells > kNoAllocMaxCells) return GRID_ERANGE;
    const uintptr_t a = reinterpret_cast<uintptr_t>(conteos);
    const uintptr_t b = reinterpret_cast<uintptr_t>(inicios);
    if (conteos == nullptr || inicios == nullptr || a % 16 || b % 16) return GRID_EINVAL;
    if (a < b + 4 * (cells + 1) && b < a + 4 * cells) return GRID_EINVAL;  // must not overlap

    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return GRID_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t tiles = ugrid::scan_tiles(cells);
    if (cudaMemsetAsync(scratch, 0, ugrid::kHeaderBytes + tiles * sizeof(unsigned long long), s) !=
        cudaSuccess)
        return GRID_ECUDA;
    auto *hdr = static_cast<grid_ws_header *>(scratch);
    auto *words =
        reinterpret_cast<unsigned long long *>(static_cast<char *>(scratch) + ugrid::kHeaderBytes);
    return ugrid::launch_scan(const_cast<uint32_t *>(conteos), inicios, cells, false, hdr, words, 1u, s,
                              false) == cudaSuccess
               ? GRID_OK
               : GRID_ECUDA;
}
