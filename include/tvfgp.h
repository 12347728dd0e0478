/*
 * tvfgp: the fast-gradient-projection (FGP) step on the dual of 3D isotropic
 * TV denoising with a nonnegativity constraint, on one NVIDIA GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no C++ or framework types.
 *
 * The operation (page "TV solver: the FGP step on the GPU", section "What one
 * step does"), for every voxel i of an nx x ny x nz volume:
 *
 *   L(r)(j) = sum_a r_a(j) - r_a(j - e_a)          (r_a(-1) = 0)
 *   z(j)    = max(b(j) - lambda L(r)(j), 0)
 *   g_a     = z(i) - z(i + e_a)                      (0 where i + e_a leaves the volume)
 *   q       = r(i) + g / (12 lambda)
 *   p'      = q / max(1, |q|)                        (|.| = Euclidean norm of the 3-vector)
 *   r(i)    = p' + m (p' - p(i));   p(i) = p'
 *
 * The momentum weight of step k is m_k = (t_k - 1) / t_{k+1} with
 * t_{k+1} = (1 + sqrt(1 + 4 t_k^2)) / 2, the FISTA schedule of the FGP method
 * (the page names only m; "Variants" and "What made the difference" describe
 * the one-kernel fused step with ping-pong r buffers that this library runs).
 *
 * Data layout (all fp32, caller-owned DEVICE memory):
 *   scalar volume (b, z):  N = nx*ny*nz floats, voxel (x,y,z) at
 *                          i = x + nx*(y + ny*z)  (x fastest);
 *   dual field (p, r):     3*N floats, planar: component a (0 = x, 1 = y,
 *                          2 = z) of voxel i at a*N + i.
 * Arithmetic: fp32, each operation rounded to nearest in the order
 *   L = ((r0(j)-r0(j-ex)) + (r1(j)-r1(j-ey))) + (r2(j)-r2(j-ez)),
 *   z = max(b - lambda*L, 0), s = fl32(1/(12*lambda)) (evaluated in double),
 *   q_a = r_a + g_a*s, |q| = sqrt((q0*q0 + q1*q1) + q2*q2), p'_a = q_a/max(1,|q|),
 *   r_a = p'_a + m*(p'_a - p_a); no fused multiply-add; IEEE division and sqrt.
 *
 * Streams: every call that touches the GPU is asynchronous on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and performs no host
 * synchronisation, except tvfgp_check().  Calls on one handle must not run
 * concurrently (the handle's scratch buffer is shared); different handles
 * are independent.
 *
 * Errors: every function returns a status code (TVFGP_OK = 0).  Argument
 * errors are detected on the host before anything is enqueued, so a failing
 * call leaves the buffers untouched.
 */
#ifndef TVFGP_H
#define TVFGP_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle: volume shape, the scratch dual buffer, the CUDA-graph cache
 * and the device error flag. */
typedef struct tvfgp_handle *tvfgp_t;

/* Same type as cudaStream_t (struct CUstream_st *), spelt without CUDA
 * headers.  NULL selects the legacy default stream. */
typedef struct CUstream_st *tvfgp_stream_t;

enum tvfgp_status {
    TVFGP_OK = 0,
    TVFGP_ERR_ARG = 1,         /* bad dimension, lambda <= 0 or not finite, nsteps < 0,
                                  NULL or aliased pointer, unknown variant/handle */
    TVFGP_ERR_ALIGN = 2,       /* a pointer is not 4-byte aligned */
    TVFGP_ERR_CUDA = 3,        /* a CUDA call failed (launch, enqueue, graph) */
    TVFGP_ERR_OOM = 4,         /* device or host allocation failed */
    TVFGP_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see tvfgp_check) */
    TVFGP_ERR_UNSUPPORTED = 6  /* the requested variant cannot run this shape/alignment */
};

/* Kernel variants.  All compute bitwise the same result. */
enum tvfgp_variant {
    TVFGP_VARIANT_AUTO = 0,      /* the measured default; falls back to SCALAR when the
                                    shape or alignment rules out the vector paths */
    TVFGP_VARIANT_FUSED = 1,     /* one kernel per step: float4 along x, the voxel's own p
                                    and r loads first, z evaluated at the voxel and at its
                                    +x, +y, +z neighbours, carried along z in registers.
                                    Needs nx % 4 == 0 and 16-byte aligned pointers. */
    TVFGP_VARIANT_SCALAR = 2,    /* one voxel per thread; any shape and alignment */
    TVFGP_VARIANT_ZMARCH_TMA = 3, /* x-y tile marching along z, planes of b, r and p staged
                                     in shared memory by TMA; same requirements as FUSED (else
                                     the call falls back to SCALAR); TVFGP_ERR_UNSUPPORTED at
                                     create/set time if the driver lacks the TMA encoder */
    TVFGP_VARIANT_ZMARCH2_TMA = 4, /* two FGP steps per pass over memory (13 volumes per two
                                     steps instead of per step), same results; used by
                                     tvfgp_run for nsteps >= 4 (a last odd step and shorter
                                     runs use ZMARCH_TMA).  The handle then owns two more
                                     buffer sets (9*nx*ny*nz more floats), allocated by
                                     tvfgp_create_ex / tvfgp_set_variant.  Same requirements
                                     as ZMARCH_TMA. */
    TVFGP_VARIANT_SEPARATE = 5,    /* the page's two-kernel step ("Variants", first row): one
                                     kernel writes z, the next reads it (18 volumes per step
                                     instead of 13); for comparison.  Any shape; the handle
                                     then owns an N-float z buffer. */
    TVFGP_VARIANT_CUBE_TMA = 6     /* the page's cube-tiled step ("Variants", 16 x 8 x 4 tile
                                     row): b and r of a 16 x 8 x 4 tile and its one-voxel halo
                                     staged in shared memory by TMA, z computed once per tile
                                     voxel; for comparison.  Same requirements as ZMARCH_TMA. */
};

/* Create a handle for an nx x ny x nz volume on the current CUDA device.
 * Allocates the scratch dual buffer (3*nx*ny*nz floats) and a device error
 * word.  1 <= nx, ny, nz <= 65535 and a plane nx*ny <= 2^31 - 1, else
 * TVFGP_ERR_ARG; the volume is bounded only by device memory.  Voxels are
 * indexed in 64 bits where nx*ny*(nz+1) exceeds 2^31 - 1 (the TMA kernels
 * always; the fused kernel through its 64-bit instance), so a run on a
 * volume of several G voxels fits the 288 GB of HBM (b, p, r and the
 * two-step path's 12 scratch volumes: 76 bytes per voxel).  *out receives
 * the handle (NULL on failure). */
int tvfgp_create(int nx, int ny, int nz, tvfgp_t *out);

/* A handle for volumes whose rows are padded: element (x, y, z) of b, of z
 * and of each component of p and r sits at x + pitch*(y + ny*z), and every
 * volume holds pitch*ny*nz elements (a dual field 3*pitch*ny*nz, component
 * a at a*pitch*ny*nz).  pitch = 2*(nx/2 + 1) is the layout of an in-place
 * real-to-complex FFT, the padded volumes of the page's solver ("Profiler
 * counters": a 256³ volume takes 64.5 MiB).  The calls read and write only
 * x < nx; the padding is never touched.  nx <= pitch <= 65535, else
 * TVFGP_ERR_ARG.  Padded rows are in general not 16-byte aligned, so the
 * float4 and TMA kernels cannot read them in place.  A tvfgp_run of 4 or more
 * steps on a handle set to AUTO, ZMARCH_TMA, ZMARCH2_TMA or CUBE_TMA with
 * nx % 4 == 0 therefore runs on dense buffers.  On AUTO and ZMARCH2_TMA
 * (with b, p, r 8-byte aligned and an even pitch) the first step reads the
 * padded rows and writes dense p, r and a dense copy of b, the dense
 * two-step kernel runs the rest, and its last launch writes p and r back
 * onto the padded rows.  The other variants pack b, p and r, run their
 * dense kernels and unpack p and r.  last_variant reports the dense
 * variant.  The handle then owns a dense handle (with its own scratch) and
 * 7*nx*ny*nz more floats, allocated on that first run (if that allocation
 * fails the run proceeds in place).  Other runs and tvfgp_step work in place: the
 * fused kernel on 8-byte halves of quads (or on pairs when nx % 4 == 2)
 * when nx and the pitch are even and b, p and r are 8-byte aligned
 * (last_variant reports FUSED), else the scalar kernel; SCALAR and SEPARATE
 * handles keep their scalar kernels.  The primal and the binary16 calls run
 * their scalar kernels.  The scratch dual is 3*pitch*ny*nz floats.
 * tvfgp_run_noalloc has no pitched form. */
int tvfgp_create_pitched(int nx, int ny, int nz, int pitch, tvfgp_t *out);

/* As tvfgp_create, choosing the kernel variant (enum tvfgp_variant).  flags
 * must be 0. */
int tvfgp_create_ex(int nx, int ny, int nz, int variant, unsigned flags, tvfgp_t *out);

/* Release the handle, its scratch buffer and cached graphs.  Waits for
 * nothing: the caller must make sure no work of this handle is in flight
 * (synchronise its streams first).  NULL is accepted. */
int tvfgp_destroy(tvfgp_t h);

/* Change the kernel variant used by later calls. */
int tvfgp_set_variant(tvfgp_t h, int variant);

/* enable != 0: tvfgp_run replays a CUDA graph of its nsteps launches (built
 * on first use for each nsteps, re-parameterised when buffers, lambda or t0
 * change); 0: launches eagerly.  Results are bitwise identical. */
int tvfgp_set_graph(tvfgp_t h, int enable);

/* Run nsteps FGP steps (sections "What one step does" and "Variants").
 *   b       [N]    device, read only: the volume being denoised;
 *   p       [3N]   device, read/write: the dual, updated in place;
 *   r       [3N]   device, read/write: the momentum copy of the dual; on
 *                  return it holds the final r (for odd nsteps the library
 *                  copies it back from its scratch buffer);
 *   lambda  > 0, finite: the TV weight;
 *   nsteps  >= 0 (0 enqueues nothing);
 *   t0      >= 1, finite: the momentum parameter t of the first step (1 for
 *           a fresh start or a restart; pass the previous *t_final to
 *           continue a run);
 *   t_final NULL or receives t after the last step (host value, available
 *           on return).
 * b, p, r and the scratch buffer must not overlap.  Asynchronous on stream.
 * The call may be recorded into the caller's CUDA graph (stream capture):
 * on a capturing stream the launches go into that graph one by one, the
 * handle's own graph is not used and nothing is allocated (a padded-row run
 * whose dense buffers do not exist yet runs in place). */
int tvfgp_run(tvfgp_t h, const float *b, float *p, float *r, float lambda, int nsteps,
              double t0, tvfgp_stream_t stream, double *t_final);

/* One FGP step with an explicit momentum weight m and explicit ping-pong
 * buffers: reads b, p, r_src; writes p (in place) and r_dst.  r_src and
 * r_dst must be distinct, non-overlapping [3N] device buffers. */
int tvfgp_step(tvfgp_t h, const float *b, float *p, const float *r_src, float *r_dst,
               float lambda, float m, tvfgp_stream_t stream);

/* The primal of a dual field, z = max(b - lambda L(dual), 0) (section "What
 * one step does", first line).  After an FGP run the denoised volume is the
 * primal of p.  b [N], dual [3N] read only; z [N] written; z must not overlap
 * b or dual. */
int tvfgp_primal(tvfgp_t h, const float *b, const float *dual, float lambda, float *z,
                 tvfgp_stream_t stream);

/* tvfgp_run with the dual stored in half precision: p and r are [3N] arrays
 * of IEEE 754 binary16 values (their bits as unsigned short), b stays fp32.
 * Each step widens the stored values exactly, computes in the fp32 canonical
 * order, and rounds each stored result once to binary16 (nearest, ties to
 * even).  It moves 28 bytes per voxel and step instead of 52 and changes the
 * result: the page ("Profiler counters") counts a half-precision dual among
 * the ways to move fewer bytes.  Kernel choice: on a handle set to
 * TVFGP_VARIANT_SCALAR the scalar kernel; on FUSED the fused vector kernel
 * when nx % 4 == 0, b is 16-byte and p, r 8-byte aligned (else scalar); on
 * every other variant the TMA z-march when nx % 8 == 0 and b, p, r are
 * 16-byte aligned, else as FUSED.  All three give the same bits;
 * tvfgp_last_variant reports ZMARCH_TMA, FUSED or SCALAR.  p and r must be
 * 2-byte aligned (TVFGP_ERR_ALIGN).  The handle's scratch buffer holds the
 * other r, so the call does not allocate. */
int tvfgp_run_f16(tvfgp_t h, const float *b, unsigned short *p, unsigned short *r, float lambda,
                  int nsteps, double t0, tvfgp_stream_t stream, double *t_final);

/* tvfgp_primal for a binary16 dual field. */
int tvfgp_primal_f16(tvfgp_t h, const float *b, const unsigned short *dual, float lambda, float *z,
                     tvfgp_stream_t stream);

/* Host only: the momentum weights m[0..nsteps-1] of a run started at t0 (in
 * double; the kernels receive each rounded once to float) and t after the
 * last step.  m may be NULL; t_final may be NULL. */
int tvfgp_momentum(double t0, int nsteps, double *m, double *t_final);

/* Synchronise `stream`, then read and clear the handle's device error word.
 * Returns TVFGP_ERR_TIMEOUT if a bounded device-side wait of an earlier call
 * gave up (its outputs are then invalid), TVFGP_ERR_CUDA if the stream
 * reports an error, else TVFGP_OK. */
int tvfgp_check(tvfgp_t h, tvfgp_stream_t stream);

/* The variant the last enqueued step actually ran (after AUTO resolution and
 * the SCALAR fallback), or -1 before the first step. */
int tvfgp_last_variant(tvfgp_t h);

/* Kernels enqueued by this handle since creation (each step, primal and
 * bounded-wait probe counts one; graph replays count their nodes). */
long long tvfgp_launch_count(tvfgp_t h);

/* Page-locked host memory for staging volumes between the host and the GPU
 * (for callers whose b comes from, or whose z goes to, host memory).  With
 * write_combined != 0 the memory is write-combined: the CPU writes it at full
 * speed and the GPU reads it at a steady rate without snooping CPU caches,
 * but CPU reads of it are very slow, so use it for host-to-device inputs
 * only.  *out receives the allocation (NULL on failure; TVFGP_ERR_OOM or
 * TVFGP_ERR_CUDA).  bytes must be > 0.  Release with tvfgp_host_free. */
int tvfgp_host_alloc(size_t bytes, int write_combined, void **out);

/* Release memory from tvfgp_host_alloc.  NULL is accepted.  The caller must
 * make sure no copy from or to it is still in flight. */
int tvfgp_host_free(void *p);

/* Test hook for the bounded-wait path: launches one block that waits on a
 * shared-memory barrier nobody arrives at, gives up after about `spins`
 * polls, sets the handle's error word and returns.  tvfgp_check() then
 * reports TVFGP_ERR_TIMEOUT.  1 <= spins <= 2^24. */
int tvfgp_debug_timeout_probe(tvfgp_t h, int spins, tvfgp_stream_t stream);

/* Test hook (no counterpart on the page): the number of polls a wait for
 * data of the TMA kernels (ZMARCH_TMA, ZMARCH2_TMA, CUBE_TMA, and the
 * binary16 z-march) makes before it gives up, for the planes of each CTA
 * from its from_plane-th on (a cube CTA has one wait, for plane 0), for
 * later calls on h (and its padded-row shadow).  polls = 0 makes those
 * waits give up at once, so a test can drive the kernels' own timeout path,
 * at the first wait (from_plane 0) or in the middle of a march with copies
 * in flight: the CTA records TVFGP_ERR_TIMEOUT in the handle's error word
 * (read by tvfgp_check), waits for its copies still in flight with the full
 * bound and returns; the outputs of that call are invalid.  polls < 0
 * restores the default (2^22 polls, and at most one second, per wait);
 * polls > 2^22 or from_plane < 0 is TVFGP_ERR_ARG.  Drops the handle's
 * cached graphs: call it with no work of h in flight. */
int tvfgp_debug_set_poll_limit(tvfgp_t h, int polls, int from_plane);

/* Test hook for allocation failures: of the library's next device
 * allocations (handle scratch, error word, extra dual sets, z volume,
 * packed staging), the first `skip` succeed and the `count` after them fail
 * with TVFGP_ERR_OOM without reaching the CUDA allocator; count = 0 clears
 * the hook.  Process-wide.  skip or count < 0: TVFGP_ERR_ARG. */
int tvfgp_debug_fail_allocs(int skip, int count);

/* Host only, no CUDA call: the launches that tvfgp_run would enqueue for a
 * run of nsteps from t0 on a handle of this shape, row pitch (0: dense) and
 * variant, given 16-byte aligned b, p, r, an available TMA encoder and
 * scratch allocations that succeed.  *route: 0 the handle's own kernels,
 * 1 a packing step and two-step launches on dense buffers (padded rows), 2
 * copies into dense buffers around a dense run and back.  *copy_back: 1 if
 * the final r is copied back from the scratch dual.  *count: the number of
 * launches; the first min(count, cap) are written as 7 ints each to items,
 * [variant, b, p_src, p_dst, r_src, r_dst, flags], and their momentum
 * weights as 2 floats each (the second one of two-step launches) to m.
 * Buffer roles: 0 b, 1 p, 2 r (the caller's), 3 the handle's scratch dual,
 * 4-6 the three dual sets of its two-step scratch, 7-9 the packed b, p and
 * r, 10 the dense handle's scratch dual, 11-13 its two-step scratch's dual
 * sets, -1 none.  flags: 1 two steps, 2 reads padded rows and writes dense
 * ones (packing step), 4 writes padded rows, 8 half of a two-kernel step.
 * Invalid shapes or arguments: TVFGP_ERR_ARG. */
int tvfgp_debug_plan(int nx, int ny, int nz, int pitch, int variant, int nsteps, double t0, int *route,
                     int *copy_back, int *items, float *m, int cap, int *count);

/* Host only, no CUDA call: how the two-step kernel splits the planes of an
 * nx x ny x nz volume among its CTAs when `slots` CTAs are resident at once
 * (SMs x CTAs per SM).  *zc: the planes of a full chunk; *count: the grid's
 * z extent; z0[j], ze[j] for j < min(count, cap): the output planes [z0, ze)
 * of the CTAs with blockIdx.z = j, by the kernel's own expressions.  Invalid
 * arguments: TVFGP_ERR_ARG. */
int tvfgp_debug_chunks(int nx, int ny, int nz, int slots, int *zc, int *z0, int *ze, int cap, int *count);

/* Self-check of the step kernels' projection onto the unit ball, which
 * evaluates q / max(1, |q|) with a hardware square-root estimate and fused
 * multiply-add corrections instead of IEEE square root and division, and
 * must give the same bits (the page's step is defined by the exact
 * operations; this check has no counterpart there).  Enqueues one kernel on
 * `stream`:
 *   mode 0: all floats nn in [1, 2^100): its square root and reciprocal
 *           against __fsqrt_rn and __frcp_rn (count is ignored);
 *   mode 1: `count` pseudo-random triples q (from `seed`): the whole
 *           projection against the IEEE one;
 *   mode 2: `count` quotients, half of them within a few ulps of a power of
 *           two, against __fdiv_rn.
 *   mode 3: `count` quads through the kernels' four-voxel update against
 *           four updates built on the IEEE projection.
 * out is a device array of two unsigned long long that the caller sets to
 * {0, ULLONG_MAX}: out[0] receives the number of mismatches, out[1] the
 * smallest mismatching sample index.  count <= 2^40; TVFGP_ERR_ARG on a bad
 * mode, count or out (NULL or not 8-byte aligned). */
int tvfgp_debug_projection_check(int mode, unsigned long long count, unsigned long long seed,
                                 unsigned long long *out, tvfgp_stream_t stream);

/* Capacity, in voxels, of tvfgp_run_noalloc's built-in scratch buffer
 * (2^21 voxels, e.g. 128^3: 3 * 2^21 floats = 24 MiB of device memory). */
#define TVFGP_NOALLOC_MAX_VOXELS 2097152

/* tvfgp_run without a handle and without any allocation.  The page has no
 * counterpart: this entry point exists for callers that must not allocate
 * device memory themselves, for example code running inside a host
 * framework that owns the whole device memory pool, a plug-in that is given
 * only buffers, or a loop that cannot afford the device-wide synchronisation
 * a cudaMalloc/cudaFree may cause.  It calls no cudaMalloc, cudaFree or other
 * allocating routine, and no host heap allocation either.
 *
 * Arguments as tvfgp_run (b [N], p and r [3N] caller-owned device buffers,
 * lambda, nsteps, t0, stream, t_final), with the shape passed directly.
 * Results are bitwise identical to tvfgp_run's.
 *
 * The second r buffer of the ping-pong is a fixed device array compiled into
 * the library (TVFGP_NOALLOC_MAX_VOXELS voxels, 24 MiB), which every GPU that
 * loads the library holds until the process exits.  Consequences:
 *   - nx*ny*nz > TVFGP_NOALLOC_MAX_VOXELS returns TVFGP_ERR_UNSUPPORTED
 *     before anything is enqueued;
 *   - all calls on one GPU share the array, which keeps the last call's
 *     contents; nothing in it needs to start at zero (each step writes every
 *     value before the next step reads it), but calls whose work overlaps on
 *     the GPU (different streams, or different host threads) race on it and
 *     must be serialised by the caller;
 *   - outside stream capture every call looks up the array's device address
 *     in the current device and context and remembers it with that
 *     context's id; a call whose stream is being captured does not look it
 *     up (the lookup may load the module) and uses the remembered address
 *     only if it belongs to the context current now.  So the first call in
 *     a context (after a cudaDeviceReset too) must come outside capture:
 *     under capture it returns TVFGP_ERR_ARG and enqueues nothing;
 *   - b, p or r overlapping the array returns TVFGP_ERR_ARG.
 * The vector kernel runs when nx % 4 == 0 and b, p, r are 16-byte aligned,
 * the scalar kernel otherwise. */
int tvfgp_run_noalloc(int nx, int ny, int nz, const float *b, float *p, float *r, float lambda,
                      int nsteps, double t0, tvfgp_stream_t stream, double *t_final);

/* Test hook (no counterpart on the page): the device address and size in
 * bytes of tvfgp_run_noalloc's built-in array on the current device, looked
 * up as an uncaptured tvfgp_run_noalloc call does.  NULL arguments:
 * TVFGP_ERR_ARG; a failed lookup: TVFGP_ERR_CUDA. */
int tvfgp_debug_noalloc_scratch(void **addr, unsigned long long *bytes);

/* Static description of a status code. */
const char *tvfgp_strerror(int code);

/* Library version, major*10000 + minor*100 + patch. */
int tvfgp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TVFGP_H */
