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
// Linear order: the three x-neighbours of a (dy, dz) row are consecutive
// cells, so each row is one range of inicios, nine ranges per particle.
// Morton order: each cell of a row has its own code; codes that follow one
// another (an even x and the x after it) are merged into one range.
// Arithmetic in fp32.
#include "ugrid_internal.cuh"

namespace ugrid {
namespace {

constexpr int kThreads = 256;

template <bool kIndirect>
__device__ __forceinline__ float accumulate(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
                                            uint32_t a, uint32_t b, float px, float py, float pz, float h2,
                                            uint32_t n, float sum) {
    b = min(b, n);
    for (uint32_t j = a; j < b; ++j) {
        const uint32_t q = kIndirect ? __ldg(ordenado + j) : j;
        if (q >= n) continue;
        const uint4 pq = __ldg(parts + 2 * (uint64_t)q);
        const float ex = __uint_as_float(pq.x) - px;
        const float ey = __uint_as_float(pq.y) - py;
        const float ez = __uint_as_float(pq.z) - pz;
        const float r2 = ex * ex + ey * ey + ez * ez;
        if (r2 < h2) {
            const float t = h2 - r2;
            const float masa =
                __uint_as_float(__ldg(reinterpret_cast<const uint32_t *>(parts) + 8 * (uint64_t)q + 7));
            sum += masa * t * t * t;
        }
    }
    return sum;
}

template <bool kIndirect, bool kMorton>
__global__ void __launch_bounds__(kThreads)
density_kernel(const uint4 *__restrict__ parts, const uint32_t *__restrict__ ordenado,
               const uint32_t *__restrict__ inicios, Geometry g, float h2, uint32_t n,
               float *__restrict__ rho, uint32_t *status) {
    allow_dependent_launch();
    grid_dependency_wait();
    const uint64_t k = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    if (k >= n) return;
    const uint32_t self = kIndirect ? __ldg(ordenado + k) : (uint32_t)k;
    if (self >= n) {
        record_status(status, kStatusBounds);
        return;
    }
    const uint4 me = __ldg(parts + 2 * (uint64_t)self);
    const float px = __uint_as_float(me.x), py = __uint_as_float(me.y), pz = __uint_as_float(me.z);
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
                                            px, py, pz, h2, n, sum);
            } else {
                uint32_t first = cell_at(x0, (uint32_t)y, (uint32_t)z, g), last = first;
                for (uint32_t x = x0 + 1; x <= x1; ++x) {
                    const uint32_t c = cell_at(x, (uint32_t)y, (uint32_t)z, g);
                    if (c != last + 1u) {
                        sum = accumulate<kIndirect>(parts, ordenado, __ldg(inicios + first), __ldg(inicios + last + 1),
                                                    px, py, pz, h2, n, sum);
                        first = c;
                    }
                    last = c;
                }
                sum = accumulate<kIndirect>(parts, ordenado, __ldg(inicios + first), __ldg(inicios + last + 1), px,
                                            py, pz, h2, n, sum);
            }
        }
    }
    rho[k] = sum;
}

}  // namespace

cudaError_t launch_density(const ugrid_particula *parts, const uint32_t *ordenado,
                           const uint32_t *inicios, const Geometry &g, float h, uint32_t n,
                           float *rho, uint32_t *status, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    const float h2 = h * h;
    const uint4 *p4 = reinterpret_cast<const uint4 *>(parts);
    const bool morton = g.order != kOrderLinear;
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
