// Neighbour density over a built grid: the consumer the grid exists for.
//
// "Construir el índice de la rejilla con un prefix sum" (§La dispersión):
// walking a cell is a loop over [inicios[c], inicios[c+1]).  "Reordenar por
// celda y la coalescencia de memoria" (§Qué cuesta la indirección, §El orden
// de las celdas): the neighbour loop visits the 27 cells around a particle;
// through ordenado every neighbour read is an indirection into origen, while
// on the reordered destino the reads are contiguous — the pages quote a 2-4x
// gain from that on SPH neighbour kernels.  For the particle at cell-order
// position k, with h <= cellSize:
//     rho[k] = sum over j with |x_j - x_k| < h of masa_j * (h^2 - r^2)^3.
// kIndirect = false reads parts (= destino) at j directly; kIndirect = true
// reads parts (= origen) at ordenado[j].  Both give the same rho[k].
//
// Linear order: one CTA per run of kTileCells cells in each of kTileRows
// consecutive y rows of one z plane (8 x 3 cells).  The candidates of all its
// particles are the particles of 3 x (kTileRows + 2) rows of cells (the own
// rows and the rows around them) over the run widened by one cell at each
// end, and in linear order each of those is one contiguous range of the cell
// order.  The CTA copies them to shared memory as (x, y, z, masa) once, then
// every thread walks the 27 cells of two particles of one cell there: three
// consecutive cells per row, nine ranges, each candidate load serving both
// particles and two candidates tested per instruction.  A run whose
// candidates do not fit falls back to the walk below.
//
// Morton order: one CTA per aligned block of up to 4 x 4 x 4 cells, its box
// of neighbour cells staged the same way (see density_morton_tile_kernel).
//
// The fallback, for a tile whose candidates do not fit and for a particle not
// in the cell it is stored in: one thread per particle walks its 27 cells in
// global memory.  In Morton order each cell of a row has its own code; codes
// that follow one another (an even x and the x after it) are merged into one
// range.
//
// Arithmetic in fp32.  A term is masa * t^3 with t = max(h^2 - r^2, 0), which
// is the term for r^2 < h^2 and an exact zero otherwise (h^2 - r^2 is formed
// by fused multiply-adds, so a candidate within an ulp or two of h can fall
// either way, at a weight of order (ulp of h^2)^3).  On the reordered records
// and through ordenado a kernel adds the same terms in the same order.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {


constexpr int kThreads = 256;
constexpr uint32_t kTileCells = 8;  // cells of one row per CTA (linear order)
// Candidates a CTA keeps in shared memory (52 KB: four CTAs per SM; an SPH
// scene of 20 particles per cell stages ~3000).
constexpr uint32_t kStageMax = 3328;
constexpr uint32_t kRowCells = kTileCells + 2;
// Threads of a tile CTA: one round over its work items, two particles each,
// ~kTileCells * kTileRows * 10 at the density of an SPH scene (a second round
// for a few threads at most); four CTAs per SM.
constexpr int kTileThreads = 288;
constexpr int kTileMinBlocks = 4;  // CTAs per SM the tile kernel is compiled for
constexpr uint32_t kTileRows = 3;  // y rows of cells per CTA
constexpr uint32_t kStagedRows = 3 * (kTileRows + 2);    // (z, y) rows whose cells are staged
static_assert(kStageMax % 2 == 0, "the linear tile stages candidates in pairs");

// sum + masa * max(h^2 - r^2, 0)^3, with h^2 - r^2 taken as three fused
// multiply-adds from h^2 and the product folded into the last add.
__device__ __forceinline__ float add_term(float sum, float4 q, float px, float py, float pz, float h2) {
    const float ex = q.x - px, ey = q.y - py, ez = q.z - pz;
    const float u = fmaf(-ez, ez, fmaf(-ey, ey, fmaf(-ex, ex, h2)));
    const float t = fmaxf(u, 0.0f);
    return fmaf(q.w * t * t, t, sum);
}

// The shared-memory tiles keep their candidates in pairs: candidates 2i and
// 2i + 1 as (x0, x1, y0, y1) and (z0, z1, w0, w1), so that one thread takes
// two candidates at a time with the packed two-lane fp32 instructions of
// sm_100 and later.  Both lanes run the arithmetic of add_term with every
// intermediate negated, which is exact under round-to-nearest: with
// v = r^2 - h^2 (= -u, the fused multiply-adds taken from -h^2) and
// m = min(v, 0) = -t, the pair adds masa * m * m * m to a running sum that is
// the negative of add_term's, and the product masa * m * m equals masa * t * t.
__device__ __forceinline__ void stage_put(float4 *st, uint32_t j, float4 q) {
    float *f = reinterpret_cast<float *>(st) + 8u * (j >> 1) + (j & 1u);
    f[0] = q.x;
    f[2] = q.y;
    f[4] = q.z;
    f[6] = q.w;
}

__device__ __forceinline__ float4 stage_get(const float4 *st, uint32_t j) {
    const float *f = reinterpret_cast<const float *>(st) + 8u * (j >> 1) + (j & 1u);
    return make_float4(f[0], f[2], f[4], f[6]);
}

// neg - masa * max(h^2 - r^2, 0)^3 for one candidate, as add_term's negative.
__device__ __forceinline__ float sub_term(float neg, float4 q, float px, float py, float pz, float nh2) {
    const float ex = q.x - px, ey = q.y - py, ez = q.z - pz;
    const float m = fminf(fmaf(ez, ez, fmaf(ey, ey, fmaf(ex, ex, nh2))), 0.0f);
    return fmaf(q.w * m * m, m, neg);
}

// Both lanes of neg for the candidate pair (a, b) = (x0, x1, y0, y1),
// (z0, z1, w0, w1); np* = the particle's coordinates negated, in both lanes.
__device__ __forceinline__ float2 sub_pair(float2 neg, float4 a, float4 b, float2 npx, float2 npy, float2 npz,
                                           float2 nh2) {
    const float2 ex = __fadd2_rn(make_float2(a.x, a.y), npx);
    const float2 ey = __fadd2_rn(make_float2(a.z, a.w), npy);
    const float2 ez = __fadd2_rn(make_float2(b.x, b.y), npz);
    float2 v = __ffma2_rn(ex, ex, nh2);
    v = __ffma2_rn(ey, ey, v);
    v = __ffma2_rn(ez, ez, v);
    const float2 m = make_float2(fminf(v.x, 0.0f), fminf(v.y, 0.0f));
    const float2 w = __fmul2_rn(__fmul2_rn(make_float2(b.z, b.w), m), m);
    return __ffma2_rn(w, m, neg);
}

// The candidates [a, b) of a paired stage added to the negated sums: an odd
// first candidate and an odd last one go to n01.x alone, pairs at even
// positions alternate between n01 and n23 in groups of four, and a last pair
// goes to n01.
__device__ __forceinline__ void walk_range(const float4 *st, uint32_t a, uint32_t b, float4 me, float2 npx,
                                           float2 npy, float2 npz, float2 nh2v, float2 &n01, float2 &n23) {
    uint32_t j = a;
    if ((j & 1u) && j < b) n01.x = sub_term(n01.x, stage_get(st, j++), me.x, me.y, me.z, nh2v.x);
    for (; j + 4 <= b; j += 4) {
        const float4 a0 = st[j], b0 = st[j + 1], a1 = st[j + 2], b1 = st[j + 3];
        n01 = sub_pair(n01, a0, b0, npx, npy, npz, nh2v);
        n23 = sub_pair(n23, a1, b1, npx, npy, npz, nh2v);
    }
    if (j + 2 <= b) {
        n01 = sub_pair(n01, st[j], st[j + 1], npx, npy, npz, nh2v);
        j += 2;
    }
    if (j < b) n01.x = sub_term(n01.x, stage_get(st, j), me.x, me.y, me.z, nh2v.x);
}

// walk_range for two particles A and B of one cell at once: each stage load
// serves both, and each particle's sums take the same terms in the same order
// as walk_range gives them.
struct PairSums {
    float2 n01, n23;
};
__device__ __forceinline__ void walk_range2(const float4 *st, uint32_t a, uint32_t b, float4 ma, float4 mb,
                                            float2 nh2v, PairSums &sa, PairSums &sb) {
    const float2 ax = make_float2(-ma.x, -ma.x), ay = make_float2(-ma.y, -ma.y), az = make_float2(-ma.z, -ma.z);
    const float2 bx = make_float2(-mb.x, -mb.x), by = make_float2(-mb.y, -mb.y), bz = make_float2(-mb.z, -mb.z);
    uint32_t j = a;
    if ((j & 1u) && j < b) {
        const float4 q = stage_get(st, j++);
        sa.n01.x = sub_term(sa.n01.x, q, ma.x, ma.y, ma.z, nh2v.x);
        sb.n01.x = sub_term(sb.n01.x, q, mb.x, mb.y, mb.z, nh2v.x);
    }
    for (; j + 4 <= b; j += 4) {
        const float4 a0 = st[j], b0 = st[j + 1], a1 = st[j + 2], b1 = st[j + 3];
        sa.n01 = sub_pair(sa.n01, a0, b0, ax, ay, az, nh2v);
        sb.n01 = sub_pair(sb.n01, a0, b0, bx, by, bz, nh2v);
        sa.n23 = sub_pair(sa.n23, a1, b1, ax, ay, az, nh2v);
        sb.n23 = sub_pair(sb.n23, a1, b1, bx, by, bz, nh2v);
    }
    if (j + 2 <= b) {
        const float4 a0 = st[j], b0 = st[j + 1];
        sa.n01 = sub_pair(sa.n01, a0, b0, ax, ay, az, nh2v);
        sb.n01 = sub_pair(sb.n01, a0, b0, bx, by, bz, nh2v);
        j += 2;
    }
    if (j < b) {
        const float4 q = stage_get(st, j);
        sa.n01.x = sub_term(sa.n01.x, q, ma.x, ma.y, ma.z, nh2v.x);
        sb.n01.x = sub_term(sb.n01.x, q, mb.x, mb.y, mb.z, nh2v.x);
    }
}

// (x, y, z, masa) of the particle at cell-order position j.
template <bool kIndirect>
__device__ __forceinline__ float4 candidate(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                            uint32_t j, uint32_t n, bool &bad) {
    const uint32_t q = kIndirect ? __ldg(ordenado + j) : j;
    if (q >= n) {
        bad = true;
        return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    const uint4 pq = __ldg(parts + 2 * (uint64_t)q);
    const float m = __uint_as_float(__ldg(reinterpret_cast<const uint32_t *>(parts) + 8 * (uint64_t)q + 7));
    return make_float4(__uint_as_float(pq.x), __uint_as_float(pq.y), __uint_as_float(pq.z), m);
}

template <bool kIndirect>
__device__ __forceinline__ float accumulate(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                            uint32_t a, uint32_t b, float px, float py, float pz, float h2,
                                            uint32_t n, float sum, uint32_t *status) {
    b = min(b, n);
    for (uint32_t j = a; j < b; ++j) {
        bool bad = false;
        const float4 q = candidate<kIndirect>(parts, ordenado, j, n, bad);
        if (bad) {
            record_status(status, kStatusBounds);
            continue;
        }
        sum = add_term(sum, q, px, py, pz, h2);
    }
    return sum;
}

// The walk in global memory for the particle at cell-order position k.
template <bool kIndirect, bool kMorton>
__device__ __forceinline__ void density_at(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                           const uint32_t *__restrict__ inicios, const Geometry &g, float h2,
                                           uint32_t n, uint32_t k, float *__restrict__ rho, uint32_t *status) {
    bool bad = false;
    const float4 me = candidate<kIndirect>(parts, ordenado, k, n, bad);
    if (bad) {
        record_status(status, kStatusBounds);
        return;
    }
    const float px = me.x, py = me.y, pz = me.z;
    const uint32_t cx = axis_coord(px, g.origin[0], g.inv_cell, g.dims[0]);
    const uint32_t cy = axis_coord(py, g.origin[1], g.inv_cell, g.dims[1]);
    const uint32_t cz = axis_coord(pz, g.origin[2], g.inv_cell, g.dims[2]);
    const uint32_t x0 = cx > 0 ? cx - 1 : 0u, x1 = cx + 1 < g.dims[0] ? cx + 1 : cx;
    float sum = 0.0f;
    for (int dz = -1; dz <= 1; ++dz) {
        const int64_t z = (int64_t)cz + dz;
        if (z < 0 || z >= (int64_t)g.dims[2]) continue;
        for (int dy = -1; dy <= 1; ++dy) {
            const int64_t y = (int64_t)cy + dy;
            if (y < 0 || y >= (int64_t)g.dims[1]) continue;
            if (!kMorton) {
                const uint64_t row = (uint64_t)g.dims[0] * ((uint64_t)y + (uint64_t)g.dims[1] * (uint64_t)z);
                sum = accumulate<kIndirect>(parts, ordenado, __ldg(inicios + row + x0), __ldg(inicios + row + x1 + 1),
                                            px, py, pz, h2, n, sum, status);
            } else {
                uint32_t first = cell_at(x0, (uint32_t)y, (uint32_t)z, g), last = first;
                for (uint32_t x = x0 + 1; x <= x1; ++x) {
                    const uint32_t c = cell_at(x, (uint32_t)y, (uint32_t)z, g);
                    if (c != last + 1u) {
                        sum = accumulate<kIndirect>(parts, ordenado, __ldg(inicios + first), __ldg(inicios + last + 1),
                                                    px, py, pz, h2, n, sum, status);
                        first = c;
                    }
                    last = c;
                }
                sum = accumulate<kIndirect>(parts, ordenado, __ldg(inicios + first), __ldg(inicios + last + 1), px,
                                            py, pz, h2, n, sum, status);
            }
        }
    }
    rho[k] = sum;
}

template <bool kIndirect, bool kMorton>
__global__ void __launch_bounds__(kThreads)
density_kernel(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
               const uint32_t *__restrict__ inicios, Geometry g, float h2, uint32_t n,
               float *__restrict__ rho, uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t k = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    if (k < n) density_at<kIndirect, kMorton>(parts, ordenado, inicios, g, h2, n, (uint32_t)k, rho, status);
}

// A tile whose candidates fit in shared memory one z plane at a time only
// (denser scenes: the pages put a healthy cell at 20 to 60 particles): the
// three planes are staged one after the other, and every work item keeps its
// two particles' sums in registers across the planes (up to kSliceRounds work
// items per thread).  Each plane's three rows give a partial sum in the same
// way as the whole tile does; the particle's density is the sum of the three
// partial sums, in plane order.  A particle not in the cell it is stored in
// takes the walk in global memory.
constexpr uint32_t kSliceRounds = 3;
template <bool kIndirect>
__device__ __forceinline__ void tile_by_planes(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                               const uint32_t *__restrict__ inicios, const Geometry &g, float h2,
                                               uint32_t n, float *__restrict__ rho, uint32_t *status,
                                               float4 *s_stage, const uint32_t (*s_start)[kRowCells + 1],
                                               const uint32_t *s_first, const uint32_t *s_items, uint32_t x0,
                                               uint32_t x1, uint32_t xa, uint32_t y0, uint32_t z, uint32_t rows) {
    const uint32_t X = g.dims[0], Y = g.dims[1], Z = g.dims[2];
    const uint32_t tid = threadIdx.x;
    const uint32_t w = x1 - x0, own_cells = rows * w, items = s_items[own_cells];
    const uint32_t nc = (x1 < X ? x1 : X - 1) - xa + 1;
    const float2 nh2v = make_float2(-h2, -h2);
    float acc[kSliceRounds][2];
#pragma unroll
    for (uint32_t rd = 0; rd < kSliceRounds; ++rd) acc[rd][0] = acc[rd][1] = 0.0f;
    for (uint32_t p = 0; p < 3; ++p) {
        const int64_t zz = (int64_t)z - 1 + (int64_t)p;
        if (zz < 0 || zz >= (int64_t)Z) continue;
        const uint32_t r0 = p * (kTileRows + 2);
        const uint32_t pbase = s_start[r0][0];
        __syncthreads();  // the previous plane's stage has been read
        for (uint32_t r = r0; r < r0 + kTileRows + 2; ++r) {
            const uint32_t base = s_start[r][0] - pbase, size = s_start[r][nc] - s_start[r][0], first = s_first[r];
            for (uint32_t j = tid; j < size; j += kTileThreads) {
                bool bad = first + j >= n;
                const float4 q = bad ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                                     : candidate<kIndirect>(parts, ordenado, first + j, n, bad);
                if (bad) record_status(status, kStatusBounds);
                stage_put(s_stage, base + j, q);
            }
        }
        __syncthreads();
#pragma unroll
        for (uint32_t rd = 0; rd < kSliceRounds; ++rd) {
            const uint32_t o = tid + rd * kTileThreads;
            if (o >= items) continue;
            uint32_t lo = 0, hi = own_cells;  // s_items[lo] <= o < s_items[hi]
            while (hi - lo > 1) {
                const uint32_t mid = (lo + hi) >> 1;
                if (s_items[mid] <= o)
                    lo = mid;
                else
                    hi = mid;
            }
            const uint32_t t = lo / w, c = (x0 - xa) + (lo - t * w), r = (kTileRows + 2) + 1 + t;
            const uint32_t s0 = s_start[r][c] + 2u * (o - s_items[lo]);
            const uint32_t s1 = s0 + 1u < s_start[r][c + 1] ? s0 + 1u : s0;
            const uint32_t ka = s_first[r] + (s0 - s_start[r][0]), kb = s_first[r] + (s1 - s_start[r][0]);
            bool bad = false;
            const float4 ma = candidate<kIndirect>(parts, ordenado, ka, n, bad);
            const float4 mb = candidate<kIndirect>(parts, ordenado, kb, n, bad);
            if (bad) continue;
            const uint32_t cx = x0 + (c - (x0 - xa)), cy = y0 + t;
            const uint32_t lo_c = (cx > 0 ? cx - 1 : 0u) - xa, hi_c = (cx + 1 < X ? cx + 1 : cx) - xa;
            PairSums sa{make_float2(-0.0f, -0.0f), make_float2(-0.0f, -0.0f)}, sb = sa;
#pragma unroll 1
            for (int dy = -1; dy <= 1; ++dy) {
                const int64_t yy = (int64_t)cy + dy;
                if (yy < 0 || yy >= (int64_t)Y) continue;
                const uint32_t rr = r0 + (t + 1 + dy);
                walk_range2(s_stage, s_start[rr][lo_c] - pbase, s_start[rr][hi_c + 1] - pbase, ma, mb, nh2v, sa, sb);
            }
            acc[rd][0] += -((sa.n01.x + sa.n01.y) + (sa.n23.x + sa.n23.y));
            acc[rd][1] += -((sb.n01.x + sb.n01.y) + (sb.n23.x + sb.n23.y));
        }
    }
#pragma unroll
    for (uint32_t rd = 0; rd < kSliceRounds; ++rd) {
        const uint32_t o = tid + rd * kTileThreads;
        if (o >= items) continue;
        uint32_t lo = 0, hi = own_cells;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (s_items[mid] <= o)
                lo = mid;
            else
                hi = mid;
        }
        const uint32_t t = lo / w, c = (x0 - xa) + (lo - t * w), r = (kTileRows + 2) + 1 + t;
        const uint32_t s0 = s_start[r][c] + 2u * (o - s_items[lo]);
        const uint32_t s1 = s0 + 1u < s_start[r][c + 1] ? s0 + 1u : s0;
        const uint32_t ka = s_first[r] + (s0 - s_start[r][0]), kb = s_first[r] + (s1 - s_start[r][0]);
        if (ka >= n || kb >= n) {
            record_status(status, kStatusBounds);
            continue;
        }
        bool bad = false;
        const float4 ma = candidate<kIndirect>(parts, ordenado, ka, n, bad);
        const float4 mb = candidate<kIndirect>(parts, ordenado, kb, n, bad);
        const uint32_t cx = x0 + (c - (x0 - xa)), cy = y0 + t;
        const bool in_a = axis_coord(ma.x, g.origin[0], g.inv_cell, X) == cx &&
                          axis_coord(ma.y, g.origin[1], g.inv_cell, Y) == cy &&
                          axis_coord(ma.z, g.origin[2], g.inv_cell, Z) == z;
        const bool in_b = axis_coord(mb.x, g.origin[0], g.inv_cell, X) == cx &&
                          axis_coord(mb.y, g.origin[1], g.inv_cell, Y) == cy &&
                          axis_coord(mb.z, g.origin[2], g.inv_cell, Z) == z;
        if (!in_a || !in_b) {
            // Not the cell they are stored in: the walk in global memory.
            density_at<kIndirect, false>(parts, ordenado, inicios, g, h2, n, ka, rho, status);
            if (s1 != s0) density_at<kIndirect, false>(parts, ordenado, inicios, g, h2, n, kb, rho, status);
            continue;
        }
        rho[ka] = acc[rd][0];
        if (s1 != s0) rho[kb] = acc[rd][1];
    }
}

// Linear order, one CTA per run of kTileCells cells of one row (see above).
template <bool kIndirect>
__global__ void __launch_bounds__(kTileThreads, kTileMinBlocks)
density_tile_kernel(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                    const uint32_t *__restrict__ inicios, Geometry g, float h2, uint32_t n,
                    float *__restrict__ rho, uint32_t *status) {
    extern __shared__ float4 s_stage[];                          // kStageMax candidates
    __shared__ uint32_t s_start[kStagedRows][kRowCells + 1];     // stage offset of each cell of each row, and the end
    __shared__ uint32_t s_first[kStagedRows];                    // cell-order index of each row's first candidate
    __shared__ uint32_t s_total;
    __shared__ uint32_t s_sliced;                                // the candidates fit plane by plane only
    __shared__ uint32_t s_items[kTileRows * kTileCells + 1];     // first work item of each own cell, and the end
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t X = g.dims[0], Y = g.dims[1], Z = g.dims[2];
    const uint32_t tiles_x = (X + kTileCells - 1) / kTileCells, tiles_y = (Y + kTileRows - 1) / kTileRows;
    const uint32_t tx = blockIdx.x % tiles_x, tyz = blockIdx.x / tiles_x;
    const uint32_t y0 = (tyz % tiles_y) * kTileRows, z = tyz / tiles_y;
    const uint32_t rows = min(kTileRows, Y - y0);                        // own rows y0 .. y0 + rows - 1
    const uint32_t x0 = tx * kTileCells, x1 = min(x0 + kTileCells, X);  // own cells [x0, x1)
    const uint32_t xa = x0 > 0 ? x0 - 1 : 0u, xb = x1 < X ? x1 : X - 1;  // staged cells [xa, xb]
    const uint32_t nc = xb - xa + 1;
    const uint32_t tid = threadIdx.x;
    // Staged row r = dzi * (kTileRows + 2) + dyi holds the cells [xa, xb] of
    // row (y0 - 1 + dyi, z - 1 + dzi), if it exists: the cells' starts,
    // relative to the row.
    for (uint32_t idx = tid; idx < kStagedRows * (nc + 1); idx += kTileThreads) {
        const uint32_t r = idx / (nc + 1), c = idx - r * (nc + 1);
        const int64_t yy = (int64_t)y0 - 1 + (int64_t)(r % (kTileRows + 2));
        const int64_t zz = (int64_t)z - 1 + (int64_t)(r / (kTileRows + 2));
        const bool exists = yy >= 0 && yy < (int64_t)Y && zz >= 0 && zz < (int64_t)Z;
        const uint64_t row = exists ? (uint64_t)X * ((uint64_t)yy + (uint64_t)Y * (uint64_t)zz) : 0;
        const uint32_t first = exists ? __ldg(inicios + row + xa) : 0u;
        s_start[r][c] = exists ? __ldg(inicios + row + xa + c) - first : 0u;
        if (c == 0) s_first[r] = first;
    }
    __syncthreads();
    static_assert(kStagedRows <= 32 && kTileRows * kTileCells <= 32, "warp 0 takes one row and one own cell per lane");
    if (tid < 32) {
        // Warp 0: lane r sums up staged row r, lane q counts the work items of
        // own cell q (rows of own cells in order, cells in order in each).
        const uint32_t lane = tid, w = x1 - x0, own = rows * w;
        uint32_t size = 0, cnt = 0;
        bool mono = true;  // starts that decrease (inconsistent input) go to the walk, too
        if (lane < kStagedRows) {
            size = s_start[lane][nc];
            for (uint32_t c = 1; c <= nc; ++c) mono &= s_start[lane][c] >= s_start[lane][c - 1];
        }
        if (lane < own) {
            // One work item per two particles of an own cell (an odd last one alone).
            const uint32_t t = lane / w, c = (x0 - xa) + (lane - t * w), r = (kTileRows + 2) + 1 + t;
            cnt = (s_start[r][c + 1] - s_start[r][c] + 1) / 2;
        }
        uint32_t base = size, first_item = cnt;  // inclusive prefixes over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t b = __shfl_up_sync(0xffffffffu, base, o), i = __shfl_up_sync(0xffffffffu, first_item, o);
            if (lane >= (uint32_t)o) {
                base += b;
                first_item += i;
            }
        }
        const uint32_t staged = __shfl_sync(0xffffffffu, base, kStagedRows - 1);
        const uint32_t items = __shfl_sync(0xffffffffu, first_item, 31);
        base -= size;
        first_item -= cnt;
        const bool row_fits = lane >= kStagedRows || (size <= kStageMax && base + size <= kStageMax);
        const bool all_mono = __all_sync(0xffffffffu, mono);
        const bool fits = __all_sync(0xffffffffu, row_fits) && all_mono;
        // Candidates of each z plane (kTileRows + 2 rows each), saturated at 2^32 - 1.
        uint64_t plane[3] = {0u, 0u, 0u};
#pragma unroll
        for (uint32_t r = 0; r < kStagedRows; ++r) plane[r / (kTileRows + 2)] += __shfl_sync(0xffffffffu, size, r);
        __syncwarp();  // every lane has read the starts before any is rebased
        if (lane < kStagedRows)
            for (uint32_t c = 0; c <= nc; ++c) s_start[lane][c] += base;
        if (lane < own) s_items[lane] = first_item;
        if (lane == 0) {
            s_items[own] = items;
            s_total = fits ? staged : 0xffffffffu;
            s_sliced = !fits && all_mono && plane[0] <= kStageMax && plane[1] <= kStageMax &&
                       plane[2] <= kStageMax && items <= kSliceRounds * kTileThreads;
        }
    }
    __syncthreads();
    const uint32_t total = s_total;
    if (total == 0xffffffffu && s_sliced) {
        tile_by_planes<kIndirect>(parts, ordenado, inicios, g, h2, n, rho, status, s_stage, s_start, s_first,
                                  s_items, x0, x1, xa, y0, z, rows);
        return;
    }
    if (total == 0xffffffffu) {
        // The candidates do not fit: each own particle walks global memory.
        for (uint32_t t = 0; t < rows; ++t) {
            const uint64_t row = (uint64_t)X * ((uint64_t)(y0 + t) + (uint64_t)Y * (uint64_t)z);
            const uint32_t k0 = __ldg(inicios + row + x0), k1 = min(__ldg(inicios + row + x1), n);
            for (uint32_t k = k0 + tid; k < k1; k += kTileThreads)
                density_at<kIndirect, false>(parts, ordenado, inicios, g, h2, n, k, rho, status);
        }
        return;
    }
    // Stage the candidates, row by row.
    for (uint32_t r = 0; r < kStagedRows; ++r) {
        const uint32_t base = s_start[r][0], size = s_start[r][nc] - base, first = s_first[r];
        for (uint32_t j = tid; j < size; j += kTileThreads) {
            bool bad = first + j >= n;
            const float4 q = bad ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                                 : candidate<kIndirect>(parts, ordenado, first + j, n, bad);
            if (bad) record_status(status, kStatusBounds);
            stage_put(s_stage, base + j, q);
        }
    }
    __syncthreads();
    // Work item o: two particles of one own cell (the last of an odd cell
    // alone), which share their 27 cells; items run over the own cells row by
    // row.
    const uint32_t w = x1 - x0, own_cells = rows * w, items = s_items[own_cells];
    for (uint32_t o = tid; o < items; o += kTileThreads) {
        uint32_t lo = 0, hi = own_cells;  // s_items[lo] <= o < s_items[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (s_items[mid] <= o)
                lo = mid;
            else
                hi = mid;
        }
        const uint32_t t = lo / w, c = (x0 - xa) + (lo - t * w), r = (kTileRows + 2) + 1 + t;
        const uint32_t s0 = s_start[r][c] + 2u * (o - s_items[lo]);
        const uint32_t s1 = s0 + 1u < s_start[r][c + 1] ? s0 + 1u : s0;  // s1 == s0: A alone
        const float4 ma = stage_get(s_stage, s0), mb = stage_get(s_stage, s1);
        const uint32_t ka = s_first[r] + (s0 - s_start[r][0]), kb = s_first[r] + (s1 - s_start[r][0]);
        const uint32_t cx = x0 + (c - (x0 - xa)), cy = y0 + t;
        const bool in_a = axis_coord(ma.x, g.origin[0], g.inv_cell, X) == cx &&
                          axis_coord(ma.y, g.origin[1], g.inv_cell, Y) == cy &&
                          axis_coord(ma.z, g.origin[2], g.inv_cell, Z) == z;
        const bool in_b = axis_coord(mb.x, g.origin[0], g.inv_cell, X) == cx &&
                          axis_coord(mb.y, g.origin[1], g.inv_cell, Y) == cy &&
                          axis_coord(mb.z, g.origin[2], g.inv_cell, Z) == z;
        if (ka >= n || kb >= n) continue;
        if (!in_a || !in_b) {
            // Not the cell they are stored in (starts inconsistent with the
            // positions): the walk in global memory, as for any order.
            density_at<kIndirect, false>(parts, ordenado, inicios, g, h2, n, ka, rho, status);
            if (s1 != s0) density_at<kIndirect, false>(parts, ordenado, inicios, g, h2, n, kb, rho, status);
            continue;
        }
        const uint32_t lo_c = (cx > 0 ? cx - 1 : 0u) - xa, hi_c = (cx + 1 < X ? cx + 1 : cx) - xa;
        const float2 nh2v = make_float2(-h2, -h2);
        PairSums sa{make_float2(-0.0f, -0.0f), make_float2(-0.0f, -0.0f)}, sb = sa;
#pragma unroll 1
        for (int dz = -1; dz <= 1; ++dz) {
            for (int dy = -1; dy <= 1; ++dy) {
                const int64_t yy = (int64_t)cy + dy, zz = (int64_t)z + dz;
                if (yy < 0 || yy >= (int64_t)Y || zz < 0 || zz >= (int64_t)Z) continue;
                const uint32_t rr = (uint32_t)(dz + 1) * (kTileRows + 2) + (t + 1 + dy);
                walk_range2(s_stage, s_start[rr][lo_c], s_start[rr][hi_c + 1], ma, mb, nh2v, sa, sb);
            }
        }
        rho[ka] = -((sa.n01.x + sa.n01.y) + (sa.n23.x + sa.n23.y));
        if (s1 != s0) rho[kb] = -((sb.n01.x + sb.n01.y) + (sb.n23.x + sb.n23.y));
    }
}


// Morton order: one CTA per aligned block of up to 4 x 4 x 4 cells.  The
// Z-curve lays out each axis's two lowest bits first, so such a block is a
// run of consecutive codes, and its particles a run of the cell order.  The
// candidates are the cells of the block widened by one cell on every side,
// each its own range of the cell order: the CTA copies them to shared memory
// (a box of up to 6 x 6 x 6 cells, x fastest, in candidate pairs), then every
// particle walks its 27 cells there as nine ranges, one per row.
constexpr uint32_t kBoxMax = 6 * 6 * 6;
constexpr uint32_t kMortonStageMax = 4608;  // candidates kept (72 KB: three CTAs per SM)
constexpr int kMortonThreads = 512;
constexpr int kMortonMinBlocks = 3;  // CTAs per SM the Morton tile kernel is compiled for
static_assert(kMortonStageMax % 2 == 0, "the Morton tile stages candidates in pairs");

__host__ __device__ __forceinline__ uint32_t morton_block_side(uint32_t dim) { return dim < 4u ? dim : 4u; }

// A Morton block whose box fits in shared memory one z plane at a time only
// (denser scenes): the box's planes are staged one after the other (each
// plane's cells are one stretch of the box order, which keeps z slowest), and
// every particle of the block (up to kMortonRounds per thread) adds, in
// registers, the rows of each plane within one cell of its own.  A particle
// not in the block's cells takes the walk in global memory.
constexpr uint32_t kMortonRounds = 8;
template <bool kIndirect>
__device__ __noinline__ void morton_by_planes(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                                 const uint32_t *__restrict__ inicios, const Geometry &g, float h2,
                                                 uint32_t n, float *__restrict__ rho, uint32_t *status,
                                                 float4 *s_stage, const uint32_t *s_box, const uint32_t *s_first,
                                                 uint32_t x0, uint32_t y0, uint32_t z0, uint32_t sx, uint32_t sy,
                                                 uint32_t sz, uint32_t xa, uint32_t ya, uint32_t za, uint32_t nx,
                                                 uint32_t ny, uint32_t nz, uint32_t k0, uint32_t k1) {
    const uint32_t X = g.dims[0], Y = g.dims[1], Z = g.dims[2];
    const uint32_t tid = threadIdx.x;
    const uint32_t per_plane = nx * ny;
    const float2 nh2v = make_float2(-h2, -h2);
    float acc[kMortonRounds];
#pragma unroll
    for (uint32_t rd = 0; rd < kMortonRounds; ++rd) acc[rd] = 0.0f;
    for (uint32_t iz = 0; iz < nz; ++iz) {
        const uint32_t c_lo = iz * per_plane, c_hi = c_lo + per_plane;
        const uint32_t pbase = s_box[c_lo], psize = s_box[c_hi] - pbase;
        const uint32_t zz = za + iz;
        __syncthreads();  // the previous plane's stage has been read
        for (uint32_t i = tid; i < psize; i += kMortonThreads) {
            uint32_t lo = c_lo, hi = c_hi;  // s_box[lo] <= pbase + i < s_box[hi]
            while (hi - lo > 1) {
                const uint32_t mid = (lo + hi) >> 1;
                if (s_box[mid] <= pbase + i)
                    lo = mid;
                else
                    hi = mid;
            }
            const uint32_t j = s_first[lo] + (pbase + i - s_box[lo]);
            bool bad = j >= n;
            const float4 q =
                bad ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : candidate<kIndirect>(parts, ordenado, j, n, bad);
            if (bad) record_status(status, kStatusBounds);
            stage_put(s_stage, i, q);
        }
        __syncthreads();
#pragma unroll
        for (uint32_t rd = 0; rd < kMortonRounds; ++rd) {
            const uint32_t k = k0 + tid + rd * kMortonThreads;
            if (k >= k1) continue;
            bool bad = false;
            const float4 me = candidate<kIndirect>(parts, ordenado, k, n, bad);
            if (bad) continue;
            const uint32_t cx = axis_coord(me.x, g.origin[0], g.inv_cell, X);
            const uint32_t cy = axis_coord(me.y, g.origin[1], g.inv_cell, Y);
            const uint32_t cz = axis_coord(me.z, g.origin[2], g.inv_cell, Z);
            if (cx < x0 || cx >= x0 + sx || cy < y0 || cy >= y0 + sy || cz < z0 || cz >= z0 + sz) continue;
            if (zz + 1 < cz || zz > cz + 1) continue;  // this plane is not one of the particle's three
            const float2 npx = make_float2(-me.x, -me.x), npy = make_float2(-me.y, -me.y);
            const float2 npz = make_float2(-me.z, -me.z);
            float2 n01 = make_float2(-0.0f, -0.0f), n23 = make_float2(-0.0f, -0.0f);
            const uint32_t xl = (cx > 0 ? cx - 1 : 0u) - xa, xh = (cx + 1 < X ? cx + 1 : cx) - xa;
#pragma unroll 1
            for (int dy = -1; dy <= 1; ++dy) {
                const int64_t yy = (int64_t)cy + dy;
                if (yy < 0 || yy >= (int64_t)Y) continue;
                const uint32_t row = c_lo + nx * ((uint32_t)yy - ya);
                walk_range(s_stage, s_box[row + xl] - pbase, s_box[row + xh + 1] - pbase, me, npx, npy, npz, nh2v,
                           n01, n23);
            }
            acc[rd] += -((n01.x + n01.y) + (n23.x + n23.y));
        }
    }
#pragma unroll
    for (uint32_t rd = 0; rd < kMortonRounds; ++rd) {
        const uint32_t k = k0 + tid + rd * kMortonThreads;
        if (k >= k1) continue;
        bool bad = false;
        const float4 me = candidate<kIndirect>(parts, ordenado, k, n, bad);
        if (bad) {
            record_status(status, kStatusBounds);
            continue;
        }
        const uint32_t cx = axis_coord(me.x, g.origin[0], g.inv_cell, X);
        const uint32_t cy = axis_coord(me.y, g.origin[1], g.inv_cell, Y);
        const uint32_t cz = axis_coord(me.z, g.origin[2], g.inv_cell, Z);
        if (cx < x0 || cx >= x0 + sx || cy < y0 || cy >= y0 + sy || cz < z0 || cz >= z0 + sz)
            density_at<kIndirect, true>(parts, ordenado, inicios, g, h2, n, k, rho, status);
        else
            rho[k] = acc[rd];
    }
}

template <bool kIndirect>
__global__ void __launch_bounds__(kMortonThreads, kMortonMinBlocks)
density_morton_tile_kernel(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                           const uint32_t *__restrict__ inicios, Geometry g, float h2, uint32_t n,
                           float *__restrict__ rho, uint32_t *status) {
    extern __shared__ float4 s_stage[];          // kMortonStageMax candidates
    __shared__ uint32_t s_box[kBoxMax + 1];      // stage offset of each box cell, and the end
    __shared__ uint32_t s_first[kBoxMax];        // cell-order index of each box cell's first particle
    __shared__ uint32_t s_total;
    __shared__ uint32_t s_sliced;                // the box fits z plane by z plane only
    allow_dependent_launch();
    grid_dependency_wait();
    const uint32_t X = g.dims[0], Y = g.dims[1], Z = g.dims[2];
    const uint32_t sx = morton_block_side(X), sy = morton_block_side(Y), sz = morton_block_side(Z);
    const uint32_t blocks_x = X / sx, blocks_y = Y / sy;
    const uint32_t bx = blockIdx.x % blocks_x, byz = blockIdx.x / blocks_x;
    const uint32_t x0 = bx * sx, y0 = (byz % blocks_y) * sy, z0 = (byz / blocks_y) * sz;
    const uint32_t xa = x0 > 0 ? x0 - 1 : 0u, ya = y0 > 0 ? y0 - 1 : 0u, za = z0 > 0 ? z0 - 1 : 0u;
    const uint32_t nx = min(x0 + sx, X - 1) - xa + 1, ny = min(y0 + sy, Y - 1) - ya + 1;
    const uint32_t nz = min(z0 + sz, Z - 1) - za + 1;
    const uint32_t ncell = nx * ny * nz;
    const uint32_t tid = threadIdx.x;
    for (uint32_t i = tid; i < ncell; i += kMortonThreads) {
        const uint32_t ix = i % nx, iy = (i / nx) % ny, iz = i / (nx * ny);
        const uint32_t c = cell_at(xa + ix, ya + iy, za + iz, g);
        const uint32_t f = __ldg(inicios + c), e = __ldg(inicios + c + 1);
        s_first[i] = f;
        s_box[i] = e >= f ? e - f : 0xffffffffu;  // starts that decrease send the block to the walk
    }
    __syncthreads();
    if (tid == 0) {
        // Offsets over the whole box while it fits; past that, offsets
        // within each z plane, as long as every plane fits (then the block
        // is staged plane by plane).
        uint32_t sum = 0;
        bool fits = true, planes = true;
        const uint32_t per_plane = nx * ny;
        for (uint32_t iz = 0; iz < nz; ++iz) {
            uint32_t psum = 0;
            for (uint32_t i = iz * per_plane; i < (iz + 1) * per_plane; ++i) {
                const uint32_t size = s_box[i];
                if (size > kMortonStageMax || psum + size > kMortonStageMax) planes = false;
                if (size > kMortonStageMax || sum + size > kMortonStageMax) fits = false;
                s_box[i] = sum;
                const uint32_t add = size > kMortonStageMax ? 0u : size;
                sum += add;
                psum += add;
            }
        }
        s_box[ncell] = sum;
        s_total = fits ? sum : 0xffffffffu;
        s_sliced = !fits && planes;
    }
    __syncthreads();
    const uint32_t total = s_total;
    const uint32_t c0 = cell_at(x0, y0, z0, g);
    const uint32_t k0 = __ldg(inicios + c0), k1 = min(__ldg(inicios + c0 + sx * sy * sz), n);
    if (total == 0xffffffffu && s_sliced && k1 >= k0 && k1 - k0 <= kMortonRounds * kMortonThreads) {
        morton_by_planes<kIndirect>(parts, ordenado, inicios, g, h2, n, rho, status, s_stage, s_box, s_first, x0,
                                    y0, z0, sx, sy, sz, xa, ya, za, nx, ny, nz, k0, k1);
        return;
    }
    if (total == 0xffffffffu) {
        for (uint32_t k = k0 + tid; k < k1; k += kMortonThreads)
            density_at<kIndirect, true>(parts, ordenado, inicios, g, h2, n, k, rho, status);
        return;
    }
    // Stage: staged index i belongs to the last box cell whose offset is <= i.
    for (uint32_t i = tid; i < total; i += kMortonThreads) {
        uint32_t lo = 0, hi = ncell;  // s_box[lo] <= i < s_box[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (s_box[mid] <= i)
                lo = mid;
            else
                hi = mid;
        }
        const uint32_t j = s_first[lo] + (i - s_box[lo]);
        bool bad = j >= n;
        const float4 q = bad ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : candidate<kIndirect>(parts, ordenado, j, n, bad);
        if (bad) record_status(status, kStatusBounds);
        stage_put(s_stage, i, q);
    }
    __syncthreads();
    for (uint32_t k = k0 + tid; k < k1; k += kMortonThreads) {
        bool bad = false;
        const float4 me = candidate<kIndirect>(parts, ordenado, k, n, bad);
        if (bad) {
            record_status(status, kStatusBounds);
            continue;
        }
        const uint32_t cx = axis_coord(me.x, g.origin[0], g.inv_cell, X);
        const uint32_t cy = axis_coord(me.y, g.origin[1], g.inv_cell, Y);
        const uint32_t cz = axis_coord(me.z, g.origin[2], g.inv_cell, Z);
        if (cx < x0 || cx >= x0 + sx || cy < y0 || cy >= y0 + sy || cz < z0 || cz >= z0 + sz) {
            density_at<kIndirect, true>(parts, ordenado, inicios, g, h2, n, k, rho, status);
            continue;
        }
        // Four negated running sums, two candidate pairs in flight.  The box
        // keeps x fastest, so the three cells of a row are one stage range.
        const float2 npx = make_float2(-me.x, -me.x), npy = make_float2(-me.y, -me.y);
        const float2 npz = make_float2(-me.z, -me.z), nh2v = make_float2(-h2, -h2);
        float2 n01 = make_float2(-0.0f, -0.0f), n23 = make_float2(-0.0f, -0.0f);
        const uint32_t xl = (cx > 0 ? cx - 1 : 0u) - xa, xh = (cx + 1 < X ? cx + 1 : cx) - xa;
#pragma unroll 1
        for (int dz = -1; dz <= 1; ++dz) {
            const int64_t zz = (int64_t)cz + dz;
            if (zz < 0 || zz >= (int64_t)Z) continue;
            for (int dy = -1; dy <= 1; ++dy) {
                const int64_t yy = (int64_t)cy + dy;
                if (yy < 0 || yy >= (int64_t)Y) continue;
                const uint32_t row = nx * (((uint32_t)yy - ya) + ny * ((uint32_t)zz - za));
                walk_range(s_stage, s_box[row + xl], s_box[row + xh + 1], me, npx, npy, npz, nh2v, n01, n23);
            }
        }
        rho[k] = -((n01.x + n01.y) + (n23.x + n23.y));
    }
}

}  // namespace

cudaError_t launch_density(const ugrid_particula *parts, const uint32_t *ordenado,
                           const uint32_t *inicios, const Geometry &g, float h, uint32_t n,
                           float *rho, uint32_t *status, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const float h2 = h * h;
    const uint4 *p4 = reinterpret_cast<const uint4 *>(parts);
    const bool morton = g.order != kOrderLinear;
    if (!morton) {
        const uint64_t tiles = (uint64_t)((g.dims[0] + kTileCells - 1) / kTileCells) *
                               ((g.dims[1] + kTileRows - 1) / kTileRows) * g.dims[2];
        const size_t smem = kStageMax * sizeof(float4);
        if (tiles <= 0x7fffffffull) {
            cudaError_t e = cudaFuncSetAttribute(ordenado ? density_tile_kernel<true> : density_tile_kernel<false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return ordenado ? launch(density_tile_kernel<true>, (unsigned)tiles, kTileThreads, smem, s, true, p4,
                                     ordenado, inicios, g, h2, n, rho, status)
                            : launch(density_tile_kernel<false>, (unsigned)tiles, kTileThreads, smem, s, true, p4,
                                     ordenado, inicios, g, h2, n, rho, status);
        }
    }
    if (morton) {
        const uint64_t blocks = (uint64_t)(g.dims[0] / morton_block_side(g.dims[0])) *
                                (g.dims[1] / morton_block_side(g.dims[1])) * (g.dims[2] / morton_block_side(g.dims[2]));
        const size_t smem = kMortonStageMax * sizeof(float4);
        if (blocks <= 0x7fffffffull) {
            cudaError_t e = cudaFuncSetAttribute(
                ordenado ? density_morton_tile_kernel<true> : density_morton_tile_kernel<false>,
                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return ordenado ? launch(density_morton_tile_kernel<true>, (unsigned)blocks, kMortonThreads, smem, s, true,
                                     p4, ordenado, inicios, g, h2, n, rho, status)
                            : launch(density_morton_tile_kernel<false>, (unsigned)blocks, kMortonThreads, smem, s, true,
                                     p4, ordenado, inicios, g, h2, n, rho, status);
        }
    }
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    if (ordenado != nullptr)
        return morton ? launch(density_kernel<true, true>, blocks, kThreads, 0, s, true, p4, ordenado, inicios, g,
                               h2, n, rho, status)
                      : launch(density_kernel<true, false>, blocks, kThreads, 0, s, true, p4, ordenado, inicios, g,
                               h2, n, rho, status);
    return morton ? launch(density_kernel<false, true>, blocks, kThreads, 0, s, true, p4, ordenado, inicios, g, h2,
                           n, rho, status)
                  : launch(density_kernel<false, false>, blocks, kThreads, 0, s, true, p4, ordenado, inicios, g, h2,
                           n, rho, status);
}

}  // namespace ugrid
