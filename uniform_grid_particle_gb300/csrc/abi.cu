// C ABI of libugrid: argument checks, workspace layout and the launch order.
// Every check runs before the first CUDA call, so a rejected call enqueues
// nothing (and works on a machine without a GPU).
#include <cmath>
#include <cstring>

#include "ugrid_internal.cuh"

namespace ugrid {

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The arrays that must be zero between calls come first, at offsets that do
// not depend on the particle count: the bucket totals (fixed size), the scan's
// look-back words and the counters (both sized by the cell count, so a call
// with fewer cells finds its words inside the ones the previous call left
// zero).  Scratch arrays sized by the particle count follow.
WsLayout ws_layout(uint64_t n, uint64_t cells, unsigned flags) {
    WsLayout l{};
    // The header's barrier and status words get 4 KB to themselves: with the
    // bucket totals right behind them, the totals' atomics slowed the
    // barrier's polling (measured: 2 us per build).
    size_t off = round_up(kHeaderBytes, 4096);
    l.bucket_total = off;
    off = round_up(off + kBucketMaxCount * kBucketLanes * sizeof(uint32_t), 256);
    l.tile_status = off;
    off = round_up(off + scan_tiles(cells) * kLookStride * sizeof(unsigned long long), 256);
    l.counts = off;
    off = round_up(off + cells * sizeof(uint32_t), 256);
    l.chunk_sums = off;
    off = round_up(off + kFusedMaxCtas * sizeof(uint32_t), 256);
    l.bucket_base = off;
    off = round_up(off + kBucketMaxCount * sizeof(uint32_t), 256);
    l.slots = off;
    off = round_up(off + n * sizeof(uint32_t), 256);
    l.pairs = off;
    off = round_up(off + n * 2 * sizeof(uint32_t), 256);
    if (flags & GRID_STABLE) {
        l.stable_queue = off;
        off = round_up(off + segment_queue_capacity(n, cells) * sizeof(uint32_t), 256);
        l.stable_scratch = off;
        off = round_up(off + n * sizeof(uint32_t), 256);
    }
    l.total = off;
    return l;
}

}  // namespace ugrid

using namespace ugrid;

namespace {

constexpr uint64_t kMaxCells = 0xfffffffeull;  // C + 1 must fit in u32

bool check_params(const grid_params *p, Geometry *g) {
    if (p == nullptr) return false;
    uint64_t c = 1;
    for (int d = 0; d < 3; ++d) {
        if (p->dims[d] == 0) return false;
        c *= p->dims[d];
        if (c > kMaxCells) return false;
    }
    if (c != p->celdas) return false;
    for (int d = 0; d < 3; ++d)
        if (!std::isfinite(p->origin[d])) return false;
    if (!std::isfinite(p->cellSize) || !(p->cellSize > 0.0f)) return false;
    const float inv = 1.0f / p->cellSize;  // fp32, rounded to nearest, once
    if (!std::isfinite(inv)) return false;
    uint32_t bits[3] = {0u, 0u, 0u};
    if (p->order == GRID_ORDER_MORTON) {
        for (int d = 0; d < 3; ++d) {
            if ((p->dims[d] & (p->dims[d] - 1u)) != 0u) return false;  // power of two
            while ((1u << bits[d]) < p->dims[d]) ++bits[d];
        }
    } else if (p->order != GRID_ORDER_LINEAR) {
        return false;
    }
    if (g != nullptr) {
        for (int d = 0; d < 3; ++d) {
            g->origin[d] = p->origin[d];
            g->dims[d] = p->dims[d];
            g->mask[d] = 0u;
        }
        g->inv_cell = inv;
        g->order = kOrderLinear;
        if (p->order == GRID_ORDER_MORTON) {
            // Walk the levels as the Z-curve lays them out and note which code
            // bit each axis's bit l lands on.
            uint32_t pos = 0u;
            for (uint32_t l = 0; l < 32u; ++l)
                for (int d = 0; d < 3; ++d)
                    if (l < bits[d]) g->mask[d] |= 1u << pos++;
            const bool cubic = bits[0] == bits[1] && bits[1] == bits[2] && bits[0] <= 10u;
            g->order = cubic ? kOrderMortonCubic : kOrderMorton;
        }
    }
    return true;
}

// An array of `count` elements: may be NULL only when empty; aligned otherwise.
bool array_ok(const void *ptr, uint64_t count, size_t align) {
    if (count == 0) return true;
    return ptr != nullptr && reinterpret_cast<uintptr_t>(ptr) % align == 0;
}

struct Span {
    const void *ptr;
    uint64_t bytes;
};

bool disjoint(const Span *s, int k) {
    for (int a = 0; a < k; ++a)
        for (int b = a + 1; b < k; ++b) {
            if (s[a].bytes == 0 || s[b].bytes == 0) continue;
            const uintptr_t pa = reinterpret_cast<uintptr_t>(s[a].ptr);
            const uintptr_t pb = reinterpret_cast<uintptr_t>(s[b].ptr);
            if (pa < pb + s[b].bytes && pb < pa + s[a].bytes) return false;
        }
    return true;
}

int cuda_code(cudaError_t e) { return e == cudaSuccess ? GRID_OK : GRID_ECUDA; }

grid_ws_header *header(void *ws) { return static_cast<grid_ws_header *>(ws); }

unsigned long long *tile_status(void *ws, const WsLayout &l) {
    return reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + l.tile_status);
}

constexpr size_t kRecord = sizeof(ugrid_particula);
static_assert(sizeof(ugrid_particula) == 32, "Particula is 32 bytes");
static_assert(offsetof(ugrid_particula, vida) == 12, "vida at byte 12");
static_assert(offsetof(ugrid_particula, vel) == 16, "vel at byte 16");
static_assert(offsetof(ugrid_particula, masa) == 28, "masa at byte 28");
static_assert(sizeof(grid_ws_header) == kHeaderBytes, "workspace header is 256 bytes");

}  // namespace

extern "C" {

size_t grid_workspace_bytes(const grid_params *p, unsigned flags) {
    if (!check_params(p, nullptr) || (flags & ~GRID_STABLE)) return 0;
    return ws_layout(p->conteo, p->celdas, flags).total;
}

int grid_workspace_init(void *ws, size_t bytes, void *stream) {
    if (ws == nullptr || bytes < kHeaderBytes || reinterpret_cast<uintptr_t>(ws) % 256) return GRID_EINVAL;
    return cuda_code(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

int grid_clear(uint32_t *conteos, const grid_params *p, void *stream) {
    if (!check_params(p, nullptr) || !array_ok(conteos, p->celdas, 16)) return GRID_EINVAL;
    return cuda_code(cudaMemsetAsync(conteos, 0, (size_t)p->celdas * sizeof(uint32_t),
                                     static_cast<cudaStream_t>(stream)));
}

int grid_count(const ugrid_particula *parts, uint32_t *conteos, uint32_t *celdaDe,
               const grid_params *p, void *stream) {
    Geometry g;
    if (!check_params(p, &g)) return GRID_EINVAL;
    const uint64_t n = p->conteo, c = p->celdas;
    if (!array_ok(parts, n, 16) || !array_ok(conteos, c, 16) || !array_ok(celdaDe, n, 4))
        return GRID_EINVAL;
    const Span s[] = {{parts, n * kRecord}, {conteos, c * 4}, {celdaDe, n * 4}};
    if (!disjoint(s, 3)) return GRID_EINVAL;
    // Launched normally: it usually follows the clear (a memset).
    return cuda_code(launch_count(parts, conteos, celdaDe, p->conteo, g,
                                  static_cast<cudaStream_t>(stream), false));
}

int grid_scan(const uint32_t *conteos, uint32_t *inicios, void *ws, const grid_params *p,
              void *stream) {
    if (!check_params(p, nullptr)) return GRID_EINVAL;
    const uint64_t c = p->celdas;
    const WsLayout l = ws_layout(p->conteo, c, 0);
    if (!array_ok(conteos, c, 16) || !array_ok(inicios, c + 1, 16) || !array_ok(ws, l.total, 256))
        return GRID_EINVAL;
    const Span s[] = {{conteos, c * 4}, {inicios, (c + 1) * 4}, {ws, l.total}};
    if (!disjoint(s, 3)) return GRID_EINVAL;
    return cuda_code(launch_scan(const_cast<uint32_t *>(conteos), inicios, c, false, header(ws),
                                 tile_status(ws, l), kLookStride, static_cast<cudaStream_t>(stream), true));
}

int grid_scatter(const uint32_t *celdaDe, const uint32_t *inicios, uint32_t *cursor,
                 uint32_t *ordenado, unsigned flags, void *ws, const grid_params *p,
                 void *stream) {
    if (!check_params(p, nullptr) || (flags & ~GRID_STABLE)) return GRID_EINVAL;
    const uint64_t n = p->conteo, c = p->celdas;
    const WsLayout l = ws_layout(n, c, flags);
    if (!array_ok(celdaDe, n, 4) || !array_ok(inicios, c + 1, 4) || !array_ok(cursor, c, 4) ||
        !array_ok(ordenado, n, 4) || !array_ok(ws, l.total, 256))
        return GRID_EINVAL;
    const Span s[] = {{celdaDe, n * 4}, {inicios, (c + 1) * 4}, {cursor, c * 4},
                      {ordenado, n * 4}, {ws, l.total}};
    if (!disjoint(s, 5)) return GRID_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    grid_ws_header *h = header(ws);
    cudaError_t e = launch_scatter(celdaDe, inicios, cursor, ordenado, p->conteo, p->celdas,
                                   &h->status, st, true);
    if (e == cudaSuccess && (flags & GRID_STABLE)) {
        char *base = static_cast<char *>(ws);
        e = launch_segment_sort(inicios, ordenado, p->conteo, p->celdas, h,
                                reinterpret_cast<uint32_t *>(base + l.stable_queue),
                                reinterpret_cast<uint32_t *>(base + l.stable_scratch), st, true);
    }
    return cuda_code(e);
}

int grid_reorder(const uint32_t *ordenado, const ugrid_particula *origen, ugrid_particula *destino,
                 void *ws, const grid_params *p, void *stream) {
    if (!check_params(p, nullptr)) return GRID_EINVAL;
    const uint64_t n = p->conteo;
    if (!array_ok(ordenado, n, 4) || !array_ok(origen, n, 16) || !array_ok(destino, n, 16) ||
        !array_ok(ws, kHeaderBytes, 256))
        return GRID_EINVAL;
    const Span s[] = {{ordenado, n * 4}, {origen, n * kRecord}, {destino, n * kRecord},
                      {ws, kHeaderBytes}};
    if (!disjoint(s, 4)) return GRID_EINVAL;
    return cuda_code(launch_reorder(ordenado, origen, destino, p->conteo, &header(ws)->status,
                                    static_cast<cudaStream_t>(stream), true));
}

int grid_build(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
               uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, void *ws,
               unsigned flags, const grid_params *p, void *stream) {
    Geometry g;
    if (!check_params(p, &g) || (flags & ~GRID_STABLE)) return GRID_EINVAL;
    const uint64_t n = p->conteo, c = p->celdas;
    const WsLayout l = ws_layout(n, c, flags);
    if (!array_ok(origen, n, 16) || !array_ok(destino, n, 16) || !array_ok(conteos, c, 16) ||
        !array_ok(celdaDe, n, 4) || !array_ok(inicios, c + 1, 16) || !array_ok(ordenado, n, 4) ||
        !array_ok(ws, l.total, 256))
        return GRID_EINVAL;
    const Span s[] = {{origen, n * kRecord}, {destino, n * kRecord}, {conteos, c * 4},
                      {celdaDe, n * 4},      {inicios, (c + 1) * 4}, {ordenado, n * 4},
                      {ws, l.total}};
    if (!disjoint(s, 7)) return GRID_EINVAL;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    grid_ws_header *h = header(ws);
    char *base = static_cast<char *>(ws);
    const bool stable = (flags & GRID_STABLE) != 0;
    if (n != 0 && !stable && n <= kClusterMaxParticles && c <= kClusterMaxCells) {
        // A small scene, non-stable: one thread-block cluster (build_cluster.cu).
        const cudaError_t f = launch_build_cluster(origen, destino, conteos, celdaDe, inicios, ordenado, (uint32_t)n,
                                                   (uint32_t)c, g, st);
        if (f != cudaErrorNotSupported) return cuda_code(f);
        (void)cudaGetLastError();
    }
    if (n != 0 && n <= kSmallMaxParticles && c <= kSmallMaxCells) {
        // A small scene: the whole build in one CTA (build_small.cu).
        return cuda_code(launch_build_small(origen, destino, conteos, celdaDe, inicios, ordenado, (uint32_t)n,
                                            (uint32_t)c, g, stable, st));
    }
    if (n != 0 && n * kSparseCellsPerParticle <= c) {
        // A sparse grid: one exchange between the particles' CTAs and the
        // cells' CTAs, one grid barrier (build_sparse.cu).
        const cudaError_t f = launch_build_sparse(
            origen, destino, conteos, celdaDe, inicios, ordenado, (uint32_t)n, c, g, h,
            reinterpret_cast<uint32_t *>(base + l.counts), reinterpret_cast<uint32_t *>(base + l.pairs), stable,
            stable ? reinterpret_cast<uint32_t *>(base + l.stable_scratch) : nullptr, st);
        if (f != cudaErrorNotSupported) return cuda_code(f);
        (void)cudaGetLastError();
    }
    if (n != 0) {
        // The two-level counting sort in one cooperative launch (build_bucketed.cu).
        const cudaError_t f = launch_build_bucketed(
            origen, destino, conteos, celdaDe, inicios, ordenado, p->conteo, c, g, h,
            reinterpret_cast<uint32_t *>(base + l.chunk_sums), reinterpret_cast<uint32_t *>(base + l.slots),
            reinterpret_cast<uint32_t *>(base + l.counts), reinterpret_cast<uint32_t *>(base + l.bucket_total),
            reinterpret_cast<uint32_t *>(base + l.bucket_base),
            reinterpret_cast<uint32_t *>(base + l.pairs), stable,
            stable ? reinterpret_cast<uint32_t *>(base + l.stable_queue) : nullptr,
            stable ? (uint32_t)segment_queue_capacity(n, c) : 0u,
            stable ? reinterpret_cast<uint32_t *>(base + l.stable_scratch) : nullptr, st);
        if (f != cudaErrorNotSupported) return cuda_code(f);
        (void)cudaGetLastError();
    }
    {
        // The whole chain in one cooperative launch (build_fused.cu).
        const cudaError_t f = launch_build_fused(
            origen, destino, conteos, celdaDe, inicios, ordenado, p->conteo, c, g, h,
            reinterpret_cast<uint32_t *>(base + l.chunk_sums),
            reinterpret_cast<uint32_t *>(base + l.slots),
            reinterpret_cast<uint32_t *>(base + l.counts), stable,
            stable ? reinterpret_cast<uint32_t *>(base + l.stable_queue) : nullptr,
            stable ? (uint32_t)segment_queue_capacity(n, c) : 0u,
            stable ? reinterpret_cast<uint32_t *>(base + l.stable_scratch) : nullptr, st);
        if (f != cudaErrorNotSupported) return cuda_code(f);
        (void)cudaGetLastError();  // not supported here: one launch per phase instead
    }
    cudaError_t e = cudaMemsetAsync(conteos, 0, c * sizeof(uint32_t), st);  // a1
    // After the memset the kernels follow one another with programmatic
    // dependent launch: each may start while the previous one drains.
    if (e == cudaSuccess) e = launch_count(origen, conteos, celdaDe, p->conteo, g, st, false);  // a2
    if (e == cudaSuccess)  // a3 and a1' (conteos zeroed tile by tile for reuse as the cursor)
        e = launch_scan(conteos, inicios, c, true, h, tile_status(ws, l), kLookStride, st, true);
    if (e == cudaSuccess)  // a4
        e = launch_scatter(celdaDe, inicios, conteos, ordenado, p->conteo, p->celdas, &h->status,
                           st, true);
    if (e == cudaSuccess && (flags & GRID_STABLE)) {  // a6
        e = launch_segment_sort(inicios, ordenado, p->conteo, p->celdas, h,
                                reinterpret_cast<uint32_t *>(base + l.stable_queue),
                                reinterpret_cast<uint32_t *>(base + l.stable_scratch), st, true);
    }
    if (e == cudaSuccess)  // a5
        e = launch_reorder(ordenado, origen, destino, p->conteo, &h->status, st, true);
    return cuda_code(e);
}

int grid_build_host(const ugrid_particula *origen_host, ugrid_particula *destino_host, uint32_t *inicios_host,
                    ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos, uint32_t *celdaDe,
                    uint32_t *inicios, uint32_t *ordenado, void *ws, unsigned flags, const grid_params *p,
                    void *stream) {
    if (!check_params(p, nullptr)) return GRID_EINVAL;
    const uint64_t n = p->conteo, c = p->celdas;
    if (inicios_host == nullptr || (n != 0 && (origen_host == nullptr || destino_host == nullptr)))
        return GRID_EINVAL;
    const Span host[] = {{origen_host, n * kRecord}, {destino_host, n * kRecord}, {inicios_host, (c + 1) * 4}};
    if (!disjoint(host, 3)) return GRID_EINVAL;
    // grid_build checks the device arrays before anything is enqueued; the
    // copy in goes first only once they have passed.
    Geometry g;
    const WsLayout l = ws_layout(n, c, flags);
    if (!check_params(p, &g) || (flags & ~GRID_STABLE) || !array_ok(origen, n, 16) || !array_ok(destino, n, 16) ||
        !array_ok(conteos, c, 16) || !array_ok(celdaDe, n, 4) || !array_ok(inicios, c + 1, 16) ||
        !array_ok(ordenado, n, 4) || !array_ok(ws, l.total, 256))
        return GRID_EINVAL;
    const Span dev[] = {{origen, n * kRecord}, {destino, n * kRecord}, {conteos, c * 4},
                        {celdaDe, n * 4},      {inicios, (c + 1) * 4}, {ordenado, n * 4},
                        {ws, l.total}};
    if (!disjoint(dev, 7)) return GRID_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n != 0) {
        const cudaError_t e = cudaMemcpyAsync(origen, origen_host, n * kRecord, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_code(e);
    }
    const int r = grid_build(origen, destino, conteos, celdaDe, inicios, ordenado, ws, flags, p, stream);
    if (r != GRID_OK) return r;
    if (n != 0) {
        const cudaError_t e = cudaMemcpyAsync(destino_host, destino, n * kRecord, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_code(e);
    }
    return cuda_code(cudaMemcpyAsync(inicios_host, inicios, (c + 1) * 4, cudaMemcpyDeviceToHost, st));
}

int grid_reorder_many(const uint32_t *ordenado, const grid_array *arrays, uint32_t count, void *ws,
                      const grid_params *p, void *stream) {
    if (!check_params(p, nullptr) || arrays == nullptr || count == 0 || count > (uint32_t)kMaxArrays)
        return GRID_EINVAL;
    const uint64_t n = p->conteo;
    if (!array_ok(ordenado, n, 4) || !array_ok(ws, kHeaderBytes, 256)) return GRID_EINVAL;
    ManyArrays m{};
    Span spans[2 + 2 * kMaxArrays];
    int k = 0;
    spans[k++] = {ordenado, n * 4};
    spans[k++] = {ws, kHeaderBytes};
    m.first[0] = 0;
    for (uint32_t a = 0; a < count; ++a) {
        const uint32_t rb = arrays[a].record_bytes;
        if (rb == 0 || rb % 16 || rb > 256) return GRID_EINVAL;
        if (!array_ok(arrays[a].origen, n, 16) || !array_ok(arrays[a].destino, n, 16)) return GRID_EINVAL;
        m.src[a] = static_cast<const uint4 *>(arrays[a].origen);
        m.dst[a] = static_cast<uint4 *>(arrays[a].destino);
        m.pieces[a] = rb / 16;
        m.first[a + 1] = m.first[a] + rb / 16;
        spans[k++] = {arrays[a].destino, n * rb};
    }
    // Destinations must not overlap each other, ordenado, the workspace, or any origen.
    if (!disjoint(spans, k)) return GRID_EINVAL;
    for (uint32_t a = 0; a < count; ++a) {
        for (uint32_t b = 0; b < count; ++b) {
            const Span pair[] = {{arrays[a].origen, n * arrays[a].record_bytes},
                                 {arrays[b].destino, n * arrays[b].record_bytes}};
            if (!disjoint(pair, 2)) return GRID_EINVAL;
        }
    }
    m.count = count;
    m.per_record = m.first[count];
    return cuda_code(launch_reorder_many(ordenado, m, p->conteo, &header(ws)->status,
                                         static_cast<cudaStream_t>(stream), true));
}

int grid_density(const ugrid_particula *parts, const uint32_t *ordenado, const uint32_t *inicios, float h,
                 float *rho, void *ws, const grid_params *p, void *stream) {
    Geometry g;
    if (!check_params(p, &g)) return GRID_EINVAL;
    if (!std::isfinite(h) || !(h > 0.0f) || h > p->cellSize) return GRID_EINVAL;
    const uint64_t n = p->conteo, c = p->celdas;
    if (!array_ok(parts, n, 16) || !array_ok(inicios, c + 1, 4) || !array_ok(rho, n, 4) ||
        !array_ok(ws, kHeaderBytes, 256) || (ordenado != nullptr && !array_ok(ordenado, n, 4)))
        return GRID_EINVAL;
    const Span s[] = {{rho, n * 4}, {parts, n * kRecord}, {inicios, (c + 1) * 4},
                      {ordenado, ordenado ? n * 4 : 0}, {ws, kHeaderBytes}};
    if (!disjoint(s, 5)) return GRID_EINVAL;
    return cuda_code(launch_density(parts, ordenado, inicios, g, h, p->conteo, rho, &header(ws)->status,
                                    static_cast<cudaStream_t>(stream)));
}

int grid_diagnostics(const uint32_t *conteos, uint32_t capacidad, uint32_t *diag,
                     const grid_params *p, void *stream) {
    if (!check_params(p, nullptr)) return GRID_EINVAL;
    const uint64_t c = p->celdas;
    if (!array_ok(conteos, c, 16) || !array_ok(diag, 2, 4)) return GRID_EINVAL;
    const Span s[] = {{conteos, c * 4}, {diag, 8}};
    if (!disjoint(s, 2)) return GRID_EINVAL;
    return cuda_code(launch_diagnostics(conteos, c, capacidad, diag, static_cast<cudaStream_t>(stream)));
}

int grid_status(void *ws, void *stream) {
    if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 256) return GRID_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GRID_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GRID_ECUDA;
    if (word != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(word), st) != cudaSuccess) return GRID_ECUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return GRID_ECUDA;
    }
    if (word & kStatusTimeout) return GRID_ETIMEOUT;
    if (word & kStatusBounds) return GRID_EBOUNDS;
    return GRID_OK;
}

const char *grid_error_string(int code) {
    switch (code) {
        case GRID_OK: return "ok";
        case GRID_EINVAL: return "invalid argument (nothing was enqueued)";
        case GRID_ECUDA: return "a CUDA call or kernel launch failed";
        case GRID_ETIMEOUT: return "a device-side wait timed out";
        case GRID_EBOUNDS: return "an index read from an input was out of range";
        case GRID_ERANGE: return "more cells than the fixed scratch of grid_scan_noalloc serves";
        default: return "unknown status code";
    }
}

}  // extern "C"
