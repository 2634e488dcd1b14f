/*
 * Uniform-grid build oracle: a plain, slow, single-threaded CPU statement of
 * what the grid build computes, written to be checked against the pages by eye.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's
 * CPU-baseline (and reference) leg load this library; the product path never
 * does, and it shares no code, header or table with the CUDA library.
 *
 * Sources (the "guia/webgpu" lessons on blog.wandres.dev):
 *   [count]   "Contar partículas por celda", §El kernel: each particle's cell
 *             index c is saved in celdaDe[i] and conteos[c] is incremented;
 *             the range guard (a clamp) lives inside the cell-index helper.
 *             §Poner a cero: conteos starts every build at zero.
 *   [scan]    "Construir el índice de la rejilla con un prefix sum",
 *             §Del conteo al inicio: inicios = exclusive scan of conteos, with
 *             one extra slot at the end holding the total.
 *   [scatter] same page, §La dispersión: a per-cell cursor starting at zero
 *             hands out slots, ordenado[inicios[c] + slot] = i;
 *             §El orden dentro de la celda: the particle index is the
 *             tie-break that makes the result reproducible.  Visiting the
 *             particles in ascending index is that order.
 *   [reorder] "Reordenar por celda y la coalescencia de memoria",
 *             §El kernel de reordenación: destino[k] = origen[ordenado[k]]
 *             (a gather of the whole 32-byte record); §El orden de las celdas:
 *             the linear cell index is x + y*GX + z*GX*GY.
 *   [record]  "El estado de las partículas en storage buffers",
 *             §La estructura y su alineación: Particula is pos (3 floats),
 *             vida, vel (3 floats), masa — 32 bytes, pos at offset 0.
 *
 * Readings where the pages are silent (the helper bodies were not on them):
 *   - cell coordinate along an axis: floor((p - o) * invCell) in fp32, with
 *     invCell = 1.0f / cellSize rounded once, each operation rounded to
 *     nearest and no fused multiply-add (build with -ffp-contract=off);
 *   - the clamp saturates to [0, dims-1]; NaN and -inf go to 0, +inf to
 *     dims-1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FLOATS_PER_PARTICLE 8
#define ORACLE_RECORD_BYTES 32

/* [count] Clamped integer cell coordinate along one axis. */
static uint32_t axis_cell(float p, float o, float invCell, uint32_t dim)
{
    float t = p - o;
    float u = t * invCell;
    float f = floorf(u);
    if (isnan(f) || f < 0.0f)
        return 0u;
    if ((double)f >= (double)dim) /* double holds every u32 exactly */
        return dim - 1u;
    return (uint32_t)f;
}

/* [reorder] §El orden de las celdas: linear index, x varies fastest. */
static uint32_t linear_cell(uint32_t x, uint32_t y, uint32_t z, uint32_t gx, uint32_t gy)
{
    return x + y * gx + z * gx * gy;
}

/* [reorder] §El orden de las celdas, the Morton (Z-curve) alternative: the
 * cell index interleaves the bits of x, y and z.  With dims = 2^bx, 2^by, 2^bz,
 * level l (from the least significant) contributes bit l of x, then of y, then
 * of z, each axis only while it still has bits; the result covers
 * [0, 2^(bx+by+bz)) exactly once. */
static uint32_t morton_cell(uint32_t x, uint32_t y, uint32_t z, const uint32_t bits[3])
{
    uint32_t code = 0u, pos = 0u;
    for (uint32_t l = 0; l < 32u; ++l) {
        if (l < bits[0]) code |= ((x >> l) & 1u) << pos++;
        if (l < bits[1]) code |= ((y >> l) & 1u) << pos++;
        if (l < bits[2]) code |= ((z >> l) & 1u) << pos++;
    }
    return code;
}

static uint32_t log2_exact(uint32_t d)
{
    uint32_t b = 0u;
    while ((1u << b) < d)
        ++b;
    return b;
}

/* Cell index of one particle's clamped coordinates in the chosen order
 * (0: linear, 1: Morton). */
static uint32_t cell_in_order(uint32_t x, uint32_t y, uint32_t z, const uint32_t dims[3], uint32_t order)
{
    if (order == 1u) {
        const uint32_t bits[3] = {log2_exact(dims[0]), log2_exact(dims[1]), log2_exact(dims[2])};
        return morton_cell(x, y, z, bits);
    }
    return linear_cell(x, y, z, dims[0], dims[1]);
}

/* Morton cell index of cell (x, y, z), exported for the pins. */
uint32_t oracle_morton_cell(uint32_t x, uint32_t y, uint32_t z, const uint32_t dims[3])
{
    return cell_in_order(x, y, z, dims, 1u);
}

/* [count] celdaDe[i] for every particle (parts: N rows of 8 floats), cells
 * numbered in `order` (0: linear, 1: Morton). */
void oracle_cell_index(const float *parts, uint64_t n, const uint32_t dims[3],
                       const float origin[3], float cellSize, uint32_t order, uint32_t *celdaDe)
{
    const float invCell = 1.0f / cellSize;
    for (uint64_t i = 0; i < n; ++i) {
        const float *pos = parts + ORACLE_FLOATS_PER_PARTICLE * i;
        uint32_t x = axis_cell(pos[0], origin[0], invCell, dims[0]);
        uint32_t y = axis_cell(pos[1], origin[1], invCell, dims[1]);
        uint32_t z = axis_cell(pos[2], origin[2], invCell, dims[2]);
        celdaDe[i] = cell_in_order(x, y, z, dims, order);
    }
}

/* [count] §Poner a cero + §El kernel: conteos = histogram of celdaDe. */
void oracle_histogram(const uint32_t *celdaDe, uint64_t n, uint32_t *conteos, uint64_t cells)
{
    memset(conteos, 0, cells * sizeof(uint32_t));
    for (uint64_t i = 0; i < n; ++i)
        conteos[celdaDe[i]] += 1u;
}

/* [scan] inicios[0] = 0, inicios[c+1] = inicios[c] + conteos[c]; C+1 entries. */
void oracle_exclusive_scan(const uint32_t *conteos, uint64_t cells, uint32_t *inicios)
{
    inicios[0] = 0u;
    for (uint64_t c = 0; c < cells; ++c)
        inicios[c + 1] = inicios[c] + conteos[c];
}

/* [scatter] Cursor scatter, particles visited in ascending index (stable). */
void oracle_scatter(const uint32_t *celdaDe, uint64_t n, const uint32_t *inicios,
                    uint32_t *cursor, uint64_t cells, uint32_t *ordenado)
{
    memset(cursor, 0, cells * sizeof(uint32_t));
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t c = celdaDe[i];
        uint32_t slot = cursor[c];
        ordenado[inicios[c] + slot] = (uint32_t)i;
        cursor[c] = slot + 1u;
    }
}

/* [reorder] destino[k] = origen[ordenado[k]], whole 32-byte records. */
void oracle_reorder(const uint32_t *ordenado, uint64_t n, const void *origen, void *destino)
{
    const unsigned char *src = (const unsigned char *)origen;
    unsigned char *dst = (unsigned char *)destino;
    for (uint64_t k = 0; k < n; ++k)
        memcpy(dst + ORACLE_RECORD_BYTES * k, src + ORACLE_RECORD_BYTES * (uint64_t)ordenado[k],
               ORACLE_RECORD_BYTES);
}

/* The whole chain: cell index, histogram, scan, scatter (stable), gather.
 * After it conteos holds the histogram again, as it does when the cursor
 * reuses the counter array and ends at the counts. */
void oracle_build(const float *origen, uint64_t n, const uint32_t dims[3], const float origin[3],
                  float cellSize, uint32_t order, uint32_t *conteos, uint32_t *celdaDe,
                  uint32_t *inicios, uint32_t *ordenado, float *destino)
{
    const uint64_t cells = (uint64_t)dims[0] * dims[1] * dims[2];
    oracle_cell_index(origen, n, dims, origin, cellSize, order, celdaDe);
    oracle_histogram(celdaDe, n, conteos, cells);
    oracle_exclusive_scan(conteos, cells, inicios);
    oracle_scatter(celdaDe, n, inicios, conteos, cells, ordenado);
    oracle_reorder(ordenado, n, origen, destino);
}

/* ---- checking helpers (not part of the method) ------------------------- */

static int cmp_u32(const void *a, const void *b)
{
    uint32_t x = *(const uint32_t *)a, y = *(const uint32_t *)b;
    return (x > y) - (x < y);
}

/* Canonical form of a cell-grouped index array: each segment
 * [inicios[c], inicios[c+1]) sorted ascending.  Order inside a cell depends
 * on scheduling ("Construir el índice…", §El orden dentro de la celda), so
 * results are compared in this form. */
void oracle_canonicalise(const uint32_t *inicios, uint64_t cells, uint32_t *ordenado)
{
    for (uint64_t c = 0; c < cells; ++c) {
        uint32_t a = inicios[c], b = inicios[c + 1];
        if (b > a + 1u)
            qsort(ordenado + a, b - a, sizeof(uint32_t), cmp_u32);
    }
}

/* [count] §Detectar el desbordamiento sin salir de la GPU: while counting,
 * previo is the counter before this particle, so previo + 1 is the cell's
 * occupancy after it; maxPorCelda keeps the largest occupancy seen and
 * desbordes counts the particles that arrive when it exceeds capacidad.
 * diag[0] = maxPorCelda, diag[1] = desbordes. */
void oracle_diagnostics(const uint32_t *celdaDe, uint64_t n, uint64_t cells, uint32_t capacidad,
                        uint32_t *cursor, uint32_t diag[2])
{
    memset(cursor, 0, cells * sizeof(uint32_t));
    diag[0] = 0u;
    diag[1] = 0u;
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t previo = cursor[celdaDe[i]];
        cursor[celdaDe[i]] = previo + 1u;
        if (previo + 1u > diag[0])
            diag[0] = previo + 1u;
        if (previo + 1u > capacidad)
            diag[1] += 1u;
    }
}

/* [reorder] §El kernel de reordenación, state in several buffers: the same
 * ordenado applied to every buffer.  For one buffer of record_bytes-byte
 * records: destino[k] = origen[ordenado[k]]; the caller applies it to each
 * buffer in turn. */
void oracle_reorder_records(const uint32_t *ordenado, uint64_t n, const void *origen, void *destino,
                            uint32_t record_bytes)
{
    const unsigned char *src = (const unsigned char *)origen;
    unsigned char *dst = (unsigned char *)destino;
    for (uint64_t k = 0; k < n; ++k)
        memcpy(dst + (uint64_t)record_bytes * k, src + (uint64_t)record_bytes * ordenado[k], record_bytes);
}

/* Neighbour density, the consumer of the grid ("Construir el índice…",
 * §La dispersión: a cell is walked as the range [inicios[c], inicios[c+1]) of
 * ordenado; "Reordenar por celda…", §Qué cuesta la indirección and §El orden
 * de las celdas: the neighbour loop visits the 27 cells around the particle).
 * With interaction radius h (h <= cellSize, so every particle closer than h
 * lies in one of the 27 cells, clamping included), for every particle i:
 *     rho[i] = sum over j with |x_j - x_i| < h of masa_j * (h^2 - |x_j - x_i|^2)^3
 * (a poly6-shaped kernel without its constant; the particle itself included),
 * evaluated in double from the fp32 records, through the indirection
 * origen[ordenado[k]], with the cells numbered in `order`. */
void oracle_density(const float *origen, uint64_t n, const uint32_t dims[3], const float origin[3],
                    float cellSize, uint32_t order, const uint32_t *inicios, const uint32_t *ordenado,
                    double h, double *rho)
{
    const float invCell = 1.0f / cellSize;
    const double h2 = h * h;
    for (uint64_t i = 0; i < n; ++i) {
        const float *pi = origen + ORACLE_FLOATS_PER_PARTICLE * i;
        const uint32_t cx = axis_cell(pi[0], origin[0], invCell, dims[0]);
        const uint32_t cy = axis_cell(pi[1], origin[1], invCell, dims[1]);
        const uint32_t cz = axis_cell(pi[2], origin[2], invCell, dims[2]);
        double sum = 0.0;
        for (int dz = -1; dz <= 1; ++dz) {
            const int64_t z = (int64_t)cz + dz;
            if (z < 0 || z >= (int64_t)dims[2])
                continue;
            for (int dy = -1; dy <= 1; ++dy) {
                const int64_t y = (int64_t)cy + dy;
                if (y < 0 || y >= (int64_t)dims[1])
                    continue;
                for (int dx = -1; dx <= 1; ++dx) {
                    const int64_t x = (int64_t)cx + dx;
                    if (x < 0 || x >= (int64_t)dims[0])
                        continue;
                    const uint32_t c = cell_in_order((uint32_t)x, (uint32_t)y, (uint32_t)z, dims, order);
                    for (uint32_t k = inicios[c]; k < inicios[c + 1]; ++k) {
                        const float *pj = origen + ORACLE_FLOATS_PER_PARTICLE * (uint64_t)ordenado[k];
                        const double ex = (double)pj[0] - (double)pi[0];
                        const double ey = (double)pj[1] - (double)pi[1];
                        const double ez = (double)pj[2] - (double)pi[2];
                        const double r2 = ex * ex + ey * ey + ez * ez;
                        if (r2 < h2) {
                            const double t = h2 - r2;
                            sum += (double)pj[7] * t * t * t;
                        }
                    }
                }
            }
        }
        rho[i] = sum;
    }
}
