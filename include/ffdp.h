/*
 * ffdp.h -- C ABI of libffdp: the fused registration objective of FFDP on one
 * GPU (sm_103a).
 *
 * Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
 * Registration" (ICLR 2026).  The entry points follow its "Key designs":
 *   item 1  fused_grid_sampler(I; A, t, [u], S, x_bounds)(x) = I(Ax + t + Su(x)),
 *           coordinates computed in registers, identity grid implicit in
 *           x_bounds, backward pass to u, A and t;
 *   item 2  Mattes mutual information with an implicit Parzen window (the
 *           B x N Parzen block is never formed; histogram entries and partial
 *           gradients accumulate in shared memory) and fused LNCC;
 *   "Background"  the objective L = C(F, M o phi) with phi(x) = Ax + t + u(x).
 *
 * Conventions shared by every call
 *   Volumes are [D][H][W] (W fastest).  Coordinates follow the PyTorch
 *   grid_sample convention: normalised [-1, 1], align_corners = true, vector
 *   components in (x, y, z) = (W, H, D) order.  Trilinear samples read 0 for
 *   taps outside the moving image.  The identity-grid coordinate of fixed
 *   voxel i along axis c is x_min[c] + (x_max[c] - x_min[c]) * i_c / (n_c - 1).
 *   A displacement u is [D][H][W][3] float32 in normalised units of M.
 *
 *   Memory: every pointer named F, M, J, u, gJ, du, dJ, dA, dt, loss, ws (and
 *   V, out, gout, dV, dR, g, m1, m2, u_out) is a DEVICE pointer owned by the
 *   caller; the library never allocates or frees device memory.
 *   ffdp_transform and the *_params structs are HOST structs read during the
 *   call.  Float and half volumes and the per-voxel vector arrays must be
 *   16-byte aligned (FFDP_ERR_INVALID_ARGUMENT otherwise).  Outputs are
 *   overwritten, never accumulated into (m1 and m2 of the optimiser step are
 *   state: read, then overwritten).
 *
 *   Streams: every call only enqueues work on `stream` (a cudaStream_t passed
 *   as void*, NULL = legacy default stream) and returns; results are ready
 *   when the stream is.  Calls on different streams may run concurrently if
 *   their workspaces and outputs are distinct.
 *
 *   Errors: arguments are validated on the host before anything is enqueued;
 *   a rejected call returns a non-zero status, launches nothing and writes
 *   nothing.  FFDP_ERR_CUDA reports a failed launch (ffdp_last_error() holds
 *   the CUDA message).  No exception crosses this interface.  No call blocks
 *   on the device.
 *
 *   Limits: each dimension in [2, 2^20]; D*H*W < 2^32 voxels; bins in [8, 64];
 *   LNCC window odd and >= 3; channels of a sampled volume in [1, 4]; a
 *   moving or sampled volume below 2^31 voxels.
 */
#ifndef FFDP_H
#define FFDP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FFDP_OK = 0,
  FFDP_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size or parameter */
  FFDP_ERR_UNSUPPORTED = 2,      /* valid request outside the built limits */
  FFDP_ERR_WORKSPACE = 3,        /* workspace missing or smaller than ffdp_workspace_bytes */
  FFDP_ERR_CUDA = 4,             /* a CUDA launch or query failed */
  FFDP_ERR_INTERNAL = 5
} ffdp_status;

typedef enum { FFDP_F32 = 0, FFDP_F16 = 1 } ffdp_dtype;

typedef struct { int64_t d, h, w; } ffdp_dims;

/* Host struct.  A and S row-major 3x3 with rows/columns in (x, y, z) order;
 * xmin/xmax are the normalised coordinates of the first and last fixed voxel
 * per axis (x_bounds; (-1, 1) for the whole moving domain). */
typedef struct {
  float A[9];
  float t[3];
  float S[9];
  float xmin[3];
  float xmax[3];
} ffdp_transform;

/* Parzen-window MI.  bins in [8, 64].  Intensities map to bin coordinates
 * c = 2 + (clamp(v, lo, hi) - lo) / (hi - lo) * (bins - 5) with the cubic
 * B-spline kernel; f_* is the fixed image's range, m_* the moving image's
 * (i.e. J's).  hi > lo required. */
typedef struct {
  int bins;
  float f_lo, f_hi, m_lo, m_hi;
} ffdp_mi_params;

/* LNCC: odd window >= 3; cc = cross^2 / (varF varJ + eps) with zero-padded
 * window sums and divisor window^3.  Windows up to 7 run in a tiled kernel
 * that keeps every window sum on chip; wider ones run as separable box sums,
 * one pass per axis, through two [5][N] float buffers of the workspace (40
 * bytes per voxel more).  A window wider than the grid sums what lies inside it. */
typedef struct {
  int window;
  float eps;
} ffdp_lncc_params;

/* Objective L = w_mi * (-MI) + w_lncc * (-LNCC).  A weight of 0 disables (does
 * not evaluate) that term; at least one weight must be non-zero. */
typedef struct {
  float w_mi, w_lncc;
  ffdp_mi_params mi;
  ffdp_lncc_params lncc;
} ffdp_objective_params;

/* Operation codes for ffdp_workspace_bytes. */
enum {
  FFDP_OP_GRID_SAMPLE_BWD = 1, /* params: NULL */
  FFDP_OP_MI = 2,              /* params: const ffdp_mi_params* */
  FFDP_OP_LNCC = 3,            /* params: const ffdp_lncc_params* */
  FFDP_OP_OBJECTIVE = 4,       /* params: const ffdp_objective_params* */
  FFDP_OP_SAMPLE_CHANNELS_BWD = 5, /* params: NULL */
  FFDP_OP_MSE = 6,             /* params: NULL */
  FFDP_OP_OBJECTIVE_MSE = 7,   /* params: NULL */
  FFDP_OP_SOBOLEV = 8,         /* params: NULL (regulariser and Adam step) */
  FFDP_OP_OBJECTIVE_STORED = 9 /* params: const ffdp_objective_params* (ffdp_objective_stored) */
};

/* Bytes of device workspace a call of `op` on fixed grid `fixed` needs (0 for
 * an invalid request).  MI and the sampler need O(bins^2 + #SMs) bytes,
 * independent of the volume size.  An objective with LNCC enabled also holds
 * the warped image J and its slope dJ/dp (16 bytes per voxel): the window
 * sums read their halo instead of re-sampling it and the sampler backward,
 * done in the backward window kernel, reads the slope instead of gathering M
 * again; the paper's fused LNCC keeps five such intermediates.  LNCC windows
 * up to 7 (the LNCC op and the objective) also hold the three g-terms the
 * forward window kernel hands to the backward one (12 bytes per voxel).  An MI-only
 * objective through ffdp_objective_stored holds the same two buffers.  An LNCC window
 * above 7 (the LNCC op or an objective with LNCC) adds 40 bytes per voxel
 * for the separable window-sum passes.  Queries the current device's SM
 * count. */
size_t ffdp_workspace_bytes(int op, ffdp_dims fixed, const void *params);

/* Design 1, forward: J[i] = M(A x_i + t + S u_i) for every fixed voxel i.
 * M: [md] volume of dtype mt; u: [out_dims][3] float32 or NULL (u = 0);
 * J_out: [out_dims] float32.  No workspace. */
ffdp_status ffdp_grid_sample_fwd(const void *M, ffdp_dtype mt, ffdp_dims mdims, ffdp_dims out_dims,
                                 const float *u, const ffdp_transform *T, float *J_out,
                                 void *stream);

/* Design 1, backward: given gJ = dL/dJ ([out_dims] float32),
 *   du_i = S^T (gJ_i dJ/dp_i),  dA = sum_i gJ_i dJ/dp_i x_i^T,  dt = sum_i gJ_i dJ/dp_i,
 * where p = A x + t + S u.  du ([out_dims][3]), dA (9, row-major) and dt (3)
 * are float32 device outputs; each may be NULL to skip it.  Workspace:
 * ffdp_workspace_bytes(FFDP_OP_GRID_SAMPLE_BWD, out_dims, NULL). */
ffdp_status ffdp_grid_sample_bwd(const void *M, ffdp_dtype mt, ffdp_dims mdims, ffdp_dims out_dims,
                                 const float *u, const ffdp_transform *T, const float *gJ,
                                 float *du, float *dA, float *dt, void *ws, size_t ws_bytes,
                                 void *stream);

/* Design 2, MI on a materialised J: loss[0] = -MI(F, J); dJ = d(-MI)/dJ
 * ([dims] float32, may be NULL).  F has dtype ft; J is float32. */
ffdp_status ffdp_mi_fwd_bwd(const void *F, ffdp_dtype ft, const float *J, ffdp_dims dims,
                            const ffdp_mi_params *p, float *loss, float *dJ, void *ws,
                            size_t ws_bytes, void *stream);

/* Design 2, LNCC on a materialised J: loss[0] = -LNCC(F, J); dJ = d(-LNCC)/dJ
 * ([dims] float32, may be NULL). */
ffdp_status ffdp_lncc_fwd_bwd(const void *F, ffdp_dtype ft, const float *J, ffdp_dims dims,
                              const ffdp_lncc_params *p, float *loss, float *dJ, void *ws,
                              size_t ws_bytes, void *stream);

/* The fused objective: J = M(Ax + t + Su) is never stored for MI; the
 * histogram sweep, the MI table, the LNCC window sums and the sampler
 * backward run as one pipeline on `stream`.
 *   loss[3] (device float32) = { w_mi*(-MI) + w_lncc*(-LNCC), -MI, -LNCC }
 *   (a disabled term reports 0);  du [fdims][3], dA[9], dt[3] as in
 *   ffdp_grid_sample_bwd (each may be NULL).  F: [fdims] of dtype ft;
 *   M: [mdims] of dtype mt. */
ffdp_status ffdp_objective(const void *F, ffdp_dtype ft, ffdp_dims fdims, const void *M,
                           ffdp_dtype mt, ffdp_dims mdims, const float *u,
                           const ffdp_transform *T, const ffdp_objective_params *p, float *loss,
                           float *du, float *dA, float *dt, void *ws, size_t ws_bytes,
                           void *stream);

/* ffdp_objective with the warped image kept for an MI-only objective: the
 * first pass also stores J and its slope dJ/dp in the workspace (16 bytes per
 * voxel, ffdp_workspace_bytes(FFDP_OP_OBJECTIVE_STORED, fdims, p)) and the
 * gradient pass streams them instead of gathering M again -- faster where the
 * memory is available (ffdp_objective keeps an MI-only objective fully
 * implicit: its workspace does not grow with the volume).  Objectives with
 * LNCC store J and its slope in either entry point, so for them the two calls
 * are the same.  Results equal ffdp_objective's up to rounding; arguments,
 * outputs and errors are as for ffdp_objective. */
ffdp_status ffdp_objective_stored(const void *F, ffdp_dtype ft, ffdp_dims fdims, const void *M,
                                  ffdp_dtype mt, ffdp_dims mdims, const float *u,
                                  const ffdp_transform *T, const ffdp_objective_params *p,
                                  float *loss, float *du, float *dA, float *dt, void *ws,
                                  size_t ws_bytes, void *stream);

/* ---- warp composition, image gradient, MSE -----------------------------
 * "Background" of the paper: the similarity C may be MSE, LNCC or MI, and
 * deformation interpolation / warp composition is one of the three memory
 * bottlenecks it profiles; design 1's sampler applies to a volume with
 * several channels unchanged, and its backward pass gives (as PyTorch's
 * grid_sample does) the gradient with respect to the sampled volume too.
 *
 * A channel-last volume V is [vdims][C] float32 (C in [1, 4], channel
 * fastest), e.g. a displacement field [D][H][W][3] like u, or the moving image
 * itself with C = 1.  p = A x + t + S u as everywhere; zero padding per tap. */

/* out[i][c] = V_c(p_i), plus (S u_i)_c when compose != 0.  compose (C = 3)
 * is warp composition: with phi(x) = A x + t + S u(x) and a second warp
 * y -> y + V(y) on V's normalised domain, V o phi composed is
 * A x + t + d(x) with d = S u + V(phi(x)) (a composite warp with S = I), and
 * out = d.  u may be NULL (u = 0); out is [out_dims][C] float32.  No
 * workspace. */
ffdp_status ffdp_sample_channels_fwd(const float *V, int C, ffdp_dims vdims, ffdp_dims out_dims,
                                     const float *u, const ffdp_transform *T, int compose, float *out,
                                     void *stream);

/* Backward of ffdp_sample_channels_fwd given gout = dL/dout ([out_dims][C]):
 *   e_i = sum_c gout_ic dV_c/dp (p_i),   du_i = S^T e_i (+ S^T gout_i if compose),
 *   dA = sum_i e_i x_i^T,  dt = sum_i e_i,
 *   dV[v][c] = sum_i gout_ic w_v(p_i)  (w_v: trilinear weight of tap v; the
 *   gradient with respect to the sampled volume -- with C = 1 and V = M, dM).
 * du ([out_dims][3]), dA (9), dt (3) and dV ([vdims][C]) may each be NULL.
 * dV is overwritten: the call zeroes it, then adds every tap's share with
 * float atomics, so its summation order (and last bits) vary between runs.
 * Workspace: ffdp_workspace_bytes(FFDP_OP_SAMPLE_CHANNELS_BWD, out_dims, NULL). */
ffdp_status ffdp_sample_channels_bwd(const float *V, int C, ffdp_dims vdims, ffdp_dims out_dims,
                                     const float *u, const ffdp_transform *T, int compose,
                                     const float *gout, float *du, float *dA, float *dt, float *dV,
                                     void *ws, size_t ws_bytes, void *stream);

/* MSE on a materialised J (design 5 calls MSE a per-voxel loss):
 * loss[0] = (1/N) sum_k (J_k - F_k)^2;  dJ = 2 (J - F) / N ([dims] float32,
 * may be NULL).  F has dtype ft; J is float32.
 * Workspace: ffdp_workspace_bytes(FFDP_OP_MSE, dims, NULL). */
ffdp_status ffdp_mse_fwd_bwd(const void *F, ffdp_dtype ft, const float *J, ffdp_dims dims, float *loss,
                             float *dJ, void *ws, size_t ws_bytes, void *stream);

/* The fused MSE objective L = w_mse * MSE(F, M o phi) in one pass over the
 * fixed grid: J = M(Ax + t + Su) and its slope are sampled in registers, the
 * per-voxel gradient 2 w_mse (J - F) / N goes straight into the sampler
 * backward; nothing per-voxel is stored.
 *   loss[2] (device float32) = { w_mse * MSE, MSE };  du [fdims][3], dA[9],
 *   dt[3] as in ffdp_grid_sample_bwd (each may be NULL).  w_mse != 0.
 * Workspace: ffdp_workspace_bytes(FFDP_OP_OBJECTIVE_MSE, fdims, NULL). */
ffdp_status ffdp_objective_mse(const void *F, ffdp_dtype ft, ffdp_dims fdims, const void *M, ffdp_dtype mt,
                               ffdp_dims mdims, const float *u, const ffdp_transform *T, float w_mse,
                               float *loss, float *du, float *dA, float *dt, void *ws, size_t ws_bytes,
                               void *stream);

/* ---- regulariser and optimiser step -----------------------------------
 * "Background": L(phi) = C(F, M o phi) + R(phi) with R a Sobolev norm; the
 * method updates the warp by gradient descent with optimiser state [m1],
 * [m2] held per voxel beside u.  The page gives no formula; these calls use
 *   R(u) = (lambda / N) sum_c sum_a sum_{i: i + e_a inside} (u_c(i + e_a) - u_c(i))^2
 * (the first-order Sobolev seminorm of u, forward differences in voxel
 * units, nothing across the boundary) and Adam with bias correction. */

/* Host struct.  step: the 1-based Adam step count t. */
typedef struct {
  float lambda;
  float lr, beta1, beta2, eps;
  int step;
} ffdp_sobolev_adam_params;

/* loss[0] = R(u); dR = dR/du = (2 lambda / N) sum_{neighbours j} (u_i - u_j)
 * ([dims][3] float32, may be NULL; must not overlap u).  u: [dims][3].
 * Workspace: ffdp_workspace_bytes(FFDP_OP_SOBOLEV, dims, NULL). */
ffdp_status ffdp_sobolev_fwd_bwd(const float *u, ffdp_dims dims, float lambda, float *loss, float *dR,
                                 void *ws, size_t ws_bytes, void *stream);

/* One regularised optimiser step of the displacement field in one pass:
 *   G = g + dR/du (g: the objective's du, e.g. from ffdp_objective),
 *   m1 = b1 m1 + (1 - b1) G,  m2 = b2 m2 + (1 - b2) G^2  (in place),
 *   u_out = u - lr (m1 / (1 - b1^t)) / (sqrt(m2 / (1 - b2^t)) + eps),
 * and loss[0] = R(u).  u, u_out, g, m1, m2 are [dims][3] float32; u_out must
 * not overlap u (the stencil reads u's neighbours: ping-pong two buffers);
 * m1 and m2 start at zero for t = 1.  The affine part (A, t: 12 numbers) is
 * left to the caller.  Workspace: ffdp_workspace_bytes(FFDP_OP_SOBOLEV, dims,
 * NULL). */
ffdp_status ffdp_sobolev_adam_step(const float *u, float *u_out, const float *g, float *m1, float *m2,
                                   ffdp_dims dims, const ffdp_sobolev_adam_params *p, float *loss, void *ws,
                                   size_t ws_bytes, void *stream);

/* Workspace-free variant of ffdp_objective for the MI term (the paper has no
 * counterpart; it exists for callers that cannot allocate device memory).
 * Some callers cannot hand the library a workspace: a plug-in inside a host
 * application that owns every device allocation, a real-time loop that may
 * not allocate after start-up, or a plain C host that only holds its input and
 * output buffers.  This entry point takes the same arguments as
 * ffdp_objective minus the workspace, and uses scratch memory reserved inside
 * the library image instead: ffdp_static_scratch_bytes() bytes (512 KiB) that
 * every GPU loading the library holds until the process exits.  It never
 * calls an allocator.
 *   - MI only and implicit, as ffdp_objective: p->w_lncc must be 0 (per-voxel
 *     images do not fit); a call whose scratch need (ffdp_workspace_bytes of
 *     the MI-only objective) exceeds the static scratch returns
 *     FFDP_ERR_UNSUPPORTED.
 *   - Each call looks up the scratch's device address on the current device
 *     (cudaGetSymbolAddress).  The first call on a device also loads the
 *     library's device code there, so make it before any stream capture;
 *     later lookups are host-side table reads.  Because nothing is cached,
 *     a cudaDeviceReset in the process needs no special handling: the next
 *     call finds the array in the new context.
 *   - All calls on a device share the one scratch area, which keeps the last
 *     call's contents; each call re-initialises what must start at zero.
 *     Calls that overlap on the GPU (e.g. on two streams at once) race on it:
 *     serialise them.
 * Outputs and errors are as for ffdp_objective. */
ffdp_status ffdp_objective_mi_static(const void *F, ffdp_dtype ft, ffdp_dims fdims, const void *M,
                                     ffdp_dtype mt, ffdp_dims mdims, const float *u,
                                     const ffdp_transform *T, const ffdp_objective_params *p,
                                     float *loss, float *du, float *dA, float *dt, void *stream);

/* Size in bytes of the static scratch used by ffdp_objective_mi_static. */
size_t ffdp_static_scratch_bytes(void);

/* Device-side failure report.  The sweep kernels stream their per-voxel
 * inputs into shared memory with asynchronous bulk copies and wait for each
 * with a time limit (1 s).  A wait that runs out marks the current device's
 * error word, the kernel finishes without touching the copies' data, and the
 * losses of that call are written as NaN (its other outputs are invalid).
 * This call synchronises the current device (the one exception to "no call
 * blocks on the device"), stores 1 in *flag if the word was marked since the
 * last call and 0 otherwise, and clears the word. */
ffdp_status ffdp_device_error(int *flag);

/* Test hook for the report above (not part of the method): when `on` is
 * non-zero, the next objective call arms the first ring slot of every warp of
 * its first sweep with 16 bytes more than the slot's copies deliver, so every
 * wait on it runs out (about two seconds in all) and the call reports through
 * ffdp_device_error and NaN losses.  Nothing faults and no copy is left in
 * flight; the request applies to one call and then clears itself. */
ffdp_status ffdp_test_ring_stall(int on);

/* Human-readable name of a status. */
const char *ffdp_status_string(ffdp_status s);

/* Detail of the last failed call on this host thread ("" if none). */
const char *ffdp_last_error(void);

/* ---- instrumentation (not part of the method) -------------------------
 * Kernel launch accounting for benchmarks: every kernel the library enqueues
 * increments a process-wide counter; when timing is enabled the library also
 * records a CUDA event pair around each launch, on the launch's own stream,
 * so per-kernel device time can be read back afterwards. */
uint64_t ffdp_launch_count(void);
/* Enable (capacity > 0: number of launches to record) or disable (0) event
 * timing.  Enabling resets previous records.  Not thread-safe with
 * concurrent library calls. */
ffdp_status ffdp_timing_enable(int capacity);
/* Synchronises the recorded events and writes, for up to `max` kernels in
 * first-launch order: a NUL-terminated name (names[k*64 ... k*64+63]), the
 * number of launches and the summed device milliseconds.  Returns the number
 * of distinct kernels (may exceed max). */
int ffdp_timing_read(char *names, int *counts, double *ms, int max);

#ifdef __cplusplus
}
#endif

#endif /* FFDP_H */
