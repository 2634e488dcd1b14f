/*
 * ugrid.h — C ABI of libugrid: a uniform spatial grid over particles, built on
 * one GB300 (sm_103a) as a counting sort keyed by cell index.
 *
 * The method is the one of the "guia/webgpu" lessons on blog.wandres.dev:
 *   "Contar partículas por celda"                       (count, clear)
 *   "Construir el índice de la rejilla con un prefix sum" (scan, scatter, order)
 *   "Reordenar por celda y la coalescencia de memoria"   (gather, cell order)
 *   "El estado de las partículas en storage buffers"     (the 32-byte record)
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     allocates no memory and keeps no state between calls (apart from what the
 *     caller's workspace holds, see grid_workspace_bytes).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream).  Nothing synchronises except grid_status.
 *   - Return value: GRID_OK when the work was enqueued; GRID_EINVAL (nothing
 *     enqueued) for a null params pointer, inconsistent params, a null or
 *     misaligned array, overlapping arrays that must be distinct, unknown flag
 *     bits; GRID_ECUDA when a CUDA call or launch failed.  Problems the GPU
 *     finds while running (a look-back wait that timed out, an index out of
 *     range) are recorded in the workspace status word and returned later by
 *     grid_status.
 *   - An empty scene (conteo = 0) is valid; every array of N elements may then
 *     be NULL.
 *   - Calls that share a workspace must not overlap on the GPU (use one
 *     workspace per concurrent stream).
 */
#ifndef UGRID_H
#define UGRID_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The particle record: pos vec3f at byte 0, vida f32 at 12, vel vec3f at 16,
 * masa f32 at 28; 32 bytes, 16-byte aligned ("El estado de las partículas en
 * storage buffers", §La estructura y su alineación).  Arrays of it are AoS. */
typedef struct ugrid_particula {
    float pos[3];
    float vida;
    float vel[3];
    float masa;
} ugrid_particula;

/* Grid geometry and sizes.  `conteo` and `celdas` are the Params uniform of
 * "Contar partículas por celda" (§El kernel); dims/origin/cellSize describe
 * the grid the cell-index helper uses.
 *   conteo    N, number of particles (0 allowed).
 *   celdas    C, number of cells; must equal dims[0]*dims[1]*dims[2] and be
 *             below 2^32 - 1 (inicios holds C + 1 u32 entries).
 *   dims      GX, GY, GZ, each >= 1.
 *   origin    lower corner of cell (0,0,0); finite.
 *   cellSize  edge of a cubic cell; finite, > 0, with 1.0f/cellSize finite.
 * Cell of a particle, per axis d (fp32, each operation rounded to nearest, no
 * fused multiply-add; invCell = 1.0f/cellSize rounded once on the host):
 *   q_d = clamp(floor((pos_d - origin_d) * invCell), 0, dims_d - 1)
 * with NaN mapped to 0 and +inf to dims_d - 1.  The cell index c follows
 * `order` ("Reordenar por celda…", §El orden de las celdas):
 *   GRID_ORDER_LINEAR  c = qx + qy*GX + qz*GX*GY (x fastest);
 *   GRID_ORDER_MORTON  the Z-curve: every side a power of two (2^bx, 2^by,
 *                      2^bz); from the least significant level l up, level l
 *                      appends bit l of qx, then of qy, then of qz, each axis
 *                      only while l is below its bit count.  The 27 cells
 *                      around a cell then span a compact range of c.
 * Every entry point that reads positions or walks cells takes the order from
 * here; a grid must be built and walked with the same order. */
typedef struct grid_params {
    uint32_t conteo;
    uint32_t celdas;
    uint32_t dims[3];
    float origin[3];
    float cellSize;
    uint32_t order; /* enum grid_order */
} grid_params;

enum grid_order {
    GRID_ORDER_LINEAR = 0u,
    GRID_ORDER_MORTON = 1u
};

enum grid_status_code {
    GRID_OK = 0,
    GRID_EINVAL = 1,   /* bad arguments; nothing was enqueued */
    GRID_ECUDA = 2,    /* a CUDA call or kernel launch failed */
    GRID_ETIMEOUT = 3, /* (grid_status) a device-side wait gave up */
    GRID_EBOUNDS = 4,  /* (grid_status) an index read from an input was out of range */
    GRID_ERANGE = 5    /* (grid_scan_noalloc) more cells than its fixed scratch serves */
};

/* flags */
enum grid_flag {
    /* Order every cell's particles by ascending particle index after the
     * scatter, so the result is reproducible bit for bit ("Construir el índice
     * de la rejilla…", §El orden dentro de la celda: particle index as the
     * tie-break).  Without it, the order inside a cell depends on scheduling. */
    GRID_STABLE = 1u
};

/* Layout of the first 256 bytes of a workspace.  Callers need not touch it;
 * it is published so that tools and tests can read the status word. */
typedef struct grid_ws_header {
    uint32_t status;       /* bit 0: a wait timed out; bit 1: an index was out of range */
    uint32_t scan_ticket;  /* next tile ticket of the running scan; 0 between calls */
    uint32_t scan_done;    /* tiles finished by the running scan; 0 between calls */
    uint32_t stable_big;   /* cells queued for the long-segment sort; 0 between calls */
    uint32_t stable_done;  /* CTAs finished by the running long-segment sort; 0 between calls */
    uint32_t bar_exit;     /* CTAs that finished the running single-launch build; 0 between calls */
    uint32_t counts_clean; /* cells of the fused build's counter array known to be zero */
    uint32_t buckets_clean; /* 1 when the bucketed build's per-bucket totals are all zero */
    uint32_t bar_extra;    /* added to every grid barrier's arrival target: 0 in use (a
                            * workspace is zero-filled); a test sets it so that the
                            * barriers' bounded waits run out */
    uint32_t reserved0[23]; /* the words above fill the first 128 bytes */
    uint32_t bar_count;    /* grid-barrier arrivals of the running single-launch build; 0 between
                            * calls.  Alone in its 128-byte line: every CTA polls it. */
    uint32_t reserved[31];
} grid_ws_header;

/* Bytes of device workspace the calls below need for these params and flags
 * (the header, the scan's per-tile look-back status words (one per 128-byte
 * line), grid_build's
 * per-CTA chunk sums, per-particle slots, per-cell counter array, per-bucket
 * totals and first positions and per-particle (cell, particle) pairs and,
 * with GRID_STABLE, the segment-sort queue and scratch).  Returns 0 for invalid
 * params.  The workspace must be 256-byte aligned and zero-filled once after
 * allocation (grid_workspace_init does that); every call leaves it ready for
 * the next one.  A workspace sized for one params/flags is valid for any
 * params with no more cells and particles and a subset of the flags. */
size_t grid_workspace_bytes(const grid_params *p, unsigned flags);

/* Zero `bytes` of workspace on `stream`. */
int grid_workspace_init(void *ws, size_t bytes, void *stream);

/* a1 — conteos[0..C) = 0, with cudaMemsetAsync ("Contar partículas por
 * celda", §Poner a cero dos millones de contadores: a fill done by the copy
 * path, ordered with the compute work).  conteos: u32[C], 16-byte aligned. */
int grid_clear(uint32_t *conteos, const grid_params *p, void *stream);

/* a2 — cell index and histogram ("Contar partículas por celda", §El kernel;
 * §La contención de las celdas densas: particles of one warp that share a cell
 * add to its counter with one atomic).  For every i < N:
 *   celdaDe[i] = cell of parts[i].pos;   conteos[celdaDe[i]] += 1.
 * parts: ugrid_particula[N], 16-byte aligned (read).  conteos: u32[C] (read
 * and written; the caller zeroes it first, e.g. with grid_clear).
 * celdaDe: u32[N], 4-byte aligned (written). */
int grid_count(const ugrid_particula *parts, uint32_t *conteos, uint32_t *celdaDe,
               const grid_params *p, void *stream);

/* a3 — exclusive scan with the total in an extra slot ("Construir el índice de
 * la rejilla…", §Del conteo al inicio):
 *   inicios[0] = 0, inicios[c+1] = inicios[c] + conteos[c], inicios[C] = N.
 * Single pass with decoupled look-back over tiles of 8192 cells.
 * conteos: u32[C] (read only).  inicios: u32[C+1] (written).  Both 16-byte
 * aligned and distinct.  ws: workspace (see grid_workspace_bytes). */
int grid_scan(const uint32_t *conteos, uint32_t *inicios, void *ws, const grid_params *p,
              void *stream);

/* a4 — cursor scatter ("Construir el índice de la rejilla…", §La dispersión):
 * for every i, slot = atomicAdd(&cursor[celdaDe[i]], 1) and
 * ordenado[inicios[celdaDe[i]] + slot] = i.  Cell c then owns
 * ordenado[inicios[c] .. inicios[c+1]).  cursor: u32[C], zero on entry (the
 * pages reuse conteos after a clear); on return it holds the histogram again.
 * celdaDe: u32[N] and inicios: u32[C+1] (read); ordenado: u32[N] (written).
 * flags: 0 or GRID_STABLE (then every segment is also sorted ascending).
 * A cell index >= C or a slot >= N read from the inputs sets status bit 1 and
 * the write is skipped. */
int grid_scatter(const uint32_t *celdaDe, const uint32_t *inicios, uint32_t *cursor,
                 uint32_t *ordenado, unsigned flags, void *ws, const grid_params *p,
                 void *stream);

/* a5 — gather reorder ("Reordenar por celda y la coalescencia de memoria",
 * §El kernel de reordenación): destino[k] = origen[ordenado[k]] for k < N,
 * whole 32-byte records; writes are contiguous, reads scattered (by the
 * tensor memory accelerator, four records per copy).
 * origen and destino are distinct, non-overlapping ugrid_particula[N] arrays,
 * 16-byte aligned.  An index >= N sets status bit 1 and that record is not
 * written.  GRID_ECUDA when the driver offers no tensor-map encoder. */
int grid_reorder(const uint32_t *ordenado, const ugrid_particula *origen, ugrid_particula *destino,
                 void *ws, const grid_params *p, void *stream);

/* The whole build: what the pages' chain computes ("Construir el índice de
 * la rejilla…", §La cadena completa: clear conteos, count, scan, clear the
 * cursor, scatter, [segment sort], gather), in one launch.  The particles are
 * first sorted into buckets of consecutive cells with shared-memory counters,
 * then each bucket's cells are counted, scanned and placed by one CTA (a
 * two-level counting sort in one cooperative launch); a bucket too large for
 * one CTA sends the launch down an atomic-counter path, and grids of more than
 * 8192 buckets use that path from the start.  Small scenes (at most 32,768
 * particles on 131,072 cells without GRID_STABLE, 8,192 on 8,192 with it) run
 * on one thread-block cluster or one CTA; sparse grids (at least four cells
 * per particle, at most 1,024 particles per CTA) exchange the particles with
 * one grid barrier.  Where a cooperative launch is not available the entry
 * points above run one after the other, the second clear folded into the
 * scan.
 * On return (once the stream has run) conteos holds the histogram, celdaDe the
 * cells, inicios the starts, ordenado the cell-grouped indices and destino
 * the reordered records; without GRID_STABLE the order inside a cell is
 * unspecified.  All seven arrays must be distinct. */
int grid_build(const ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos,
               uint32_t *celdaDe, uint32_t *inicios, uint32_t *ordenado, void *ws,
               unsigned flags, const grid_params *p, void *stream);

/* grid_build from and to host memory, all on `stream`: origen_host (N records)
 * is copied into the device array origen, the grid is built exactly as by
 * grid_build, then destino and inicios are copied back into destino_host
 * (N records) and inicios_host (C+1 words).  The host arrays should be
 * page-locked (cudaHostAlloc / cudaHostRegister) for the copies to be
 * asynchronous; they must not overlap each other.  The device arrays follow
 * grid_build's rules.  The host results are complete once the stream has run
 * (synchronise it, or wait on an event recorded after the call).  Returns
 * GRID_EINVAL for a null host array when N > 0 (inicios_host always), else
 * what the copies and grid_build return. */
int grid_build_host(const ugrid_particula *origen_host, ugrid_particula *destino_host, uint32_t *inicios_host,
                    ugrid_particula *origen, ugrid_particula *destino, uint32_t *conteos, uint32_t *celdaDe,
                    uint32_t *inicios, uint32_t *ordenado, void *ws, unsigned flags, const grid_params *p,
                    void *stream);

/* Exclusive scan for callers that cannot allocate device memory; the pages
 * have no counterpart to it.  It computes exactly what grid_scan computes
 * (inicios[0] = 0, inicios[c+1] = inicios[c] + conteos[c], inicios[C] = N),
 * but keeps the scan's scratch — a 256-byte header and one 64-bit look-back
 * word per 8192-cell tile — in a fixed 33,024-byte array inside the library
 * instead of a caller workspace.  It is meant for code that may not take
 * device memory itself: an engine that owns every device buffer and hands
 * them out from its own pool, or a per-frame step that cannot risk cudaMalloc
 * stalling the device.  It allocates nothing and calls no allocating routine.
 *   conteos  u32[C], read only; inicios u32[C+1], written; both device
 *            pointers, 16-byte aligned, not overlapping.
 *   p        as for grid_scan; celdas must be at most 33,554,432 (4096 tiles),
 *            otherwise GRID_ERANGE is returned and nothing is enqueued.
 * Returns GRID_OK, GRID_EINVAL (bad params or arrays, nothing enqueued),
 * GRID_ERANGE, or GRID_ECUDA.  The first call on each device (with that
 * device current) looks up the array's device address and caches it with the
 * current context; make that first call before capturing any stream.  After
 * the device's context is destroyed and created again (cudaDeviceReset), the
 * next call finds a new context and looks the address up again, so that call
 * too should come before any capture.  All calls share the one
 * array, which each call clears on its stream before use: calls whose work
 * overlaps on the GPU race on it and must be ordered by the caller.  A
 * device-side wait that gives up is recorded only in that array and is not
 * reported: a caller that needs to detect it uses grid_scan with a workspace
 * and grid_status. */
int grid_scan_noalloc(const uint32_t *conteos, uint32_t *inicios, const grid_params *p,
                      void *stream);

/* One particle array for grid_reorder_many: device pointers to N records of
 * record_bytes bytes each (a multiple of 16, at most 256), 16-byte aligned. */
typedef struct grid_array {
    const void *origen;
    void *destino;
    uint32_t record_bytes;
} grid_array;

/* Gather several arrays with one ordenado ("Reordenar por celda…", §El kernel
 * de reordenación: when the state lives in several buffers, one kernel that
 * reads ordenado[k] once for all of them beats one kernel per buffer; "El
 * estado de las partículas…", §AoS o SoA: the hot/cold split).  For every
 * array a and k < N: destino_a[k] = origen_a[ordenado[k]].
 * arrays: host array of `count` descriptors, 1 <= count <= 4.  Every destino
 * must be distinct from every origen and destino, ordenado and the workspace
 * header.  An index >= N sets status bit 1 (see grid_status) and that record
 * is not written. */
int grid_reorder_many(const uint32_t *ordenado, const grid_array *arrays, uint32_t count, void *ws,
                      const grid_params *p, void *stream);

/* Neighbour density, the query the grid is built for ("Construir el índice…",
 * §La dispersión: a cell is the range [inicios[c], inicios[c+1]) of the
 * cell order; "Reordenar por celda…", §Qué cuesta la indirección and §El
 * orden de las celdas: the neighbour loop visits the 27 cells around the
 * particle).  For the particle at cell-order position k and radius h:
 *   rho[k] = sum over particles j with |x_j - x_k| < h of
 *            masa_j * (h^2 - |x_j - x_k|^2)^3        (itself included)
 * in fp32.  Two ways to read the particles, with the same result:
 *   ordenado == NULL  parts is the reordered destino of a build (contiguous
 *                     reads, the point of the reorder);
 *   ordenado != NULL  parts is the original origen, read at ordenado[j]
 *                     (the indirection the reorder removes).
 * inicios: u32[C+1] of the same build.  rho: float[N] (written).
 * 0 < h <= cellSize (so the 27 cells hold every neighbour), else GRID_EINVAL.
 * An index >= N read from ordenado sets status bit 1 and is skipped. */
int grid_density(const ugrid_particula *parts, const uint32_t *ordenado, const uint32_t *inicios, float h,
                 float *rho, void *ws, const grid_params *p, void *stream);

/* Overflow diagnostics ("Contar partículas por celda", §Detectar el
 * desbordamiento sin salir de la GPU): for a per-cell capacity, the largest
 * occupancy (maxPorCelda: the page's atomicMax of previo + 1 while counting)
 * and the number of particles that arrived over the capacity (desbordes).
 * Both are fixed by the histogram, so they are computed from it in one pass:
 *   diag[0] = max_c conteos[c],  diag[1] = sum_c max(0, conteos[c] - capacidad).
 * conteos: u32[C] (read), 16-byte aligned, e.g. as left by grid_count or
 * grid_build.  diag: u32[2] device array (written; zeroed first on `stream`).
 * The page uses capacidad = 64. */
int grid_diagnostics(const uint32_t *conteos, uint32_t capacidad, uint32_t *diag,
                     const grid_params *p, void *stream);

/* Synchronise `stream`, read and clear the workspace status word, and return
 * GRID_OK, GRID_ETIMEOUT (bit 0 set) or GRID_EBOUNDS (bit 1 set); GRID_ECUDA
 * if the copy or the synchronisation failed. */
int grid_status(void *ws, void *stream);

/* Static description of a status code (never NULL). */
const char *grid_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* UGRID_H */
