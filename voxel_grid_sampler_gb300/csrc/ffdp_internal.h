// ffdp_internal.h -- argument records and launcher declarations shared by the
// host ABI (ffdp_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "ffdp_device.cuh"

// Instantiate a body for the float (code 0) or half (code 1) element type.
#define FFDP_DT_SWITCH(code, T, ...)      \
  do {                                    \
    if ((code) == 0) {                    \
      using T = float;                    \
      __VA_ARGS__;                        \
    } else {                              \
      using T = __half;                   \
      __VA_ARGS__;                        \
    }                                     \
  } while (0)

namespace ffdp {

// Sweep 1: histogram; + J store; J store only; histogram of a given J;
// histogram + J and dJ/dq stores; J and dJ/dq stores only.
enum Sweep1Mode { S1_HIST = 0, S1_HIST_WRITEJ = 1, S1_WRITEJ = 2, S1_HIST_JBUF = 3, S1_HIST_WRITEJG = 4, S1_WRITEJG = 5 };
constexpr int kSweep1Modes = 6;
// Sweep 2: MI gradient + sampler backward; sampler backward of a given g;
// MI gradient of a given J; backward of a given g with the stored dJ/dq (no
// gathers); MI gradient + backward from the stored J and dJ/dq (no gathers);
// MSE gradient 2 w (J - F) / N + backward, one pass (gathers).
enum Sweep2Mode { S2_MI = 0, S2_GBUF = 1, S2_MI_JBUF = 2, S2_GBUF_DJ = 3, S2_MI_DJ = 4, S2_MSE = 5 };
// threads per CTA of a gradient-sweep mode: the gathering modes at
// kSweep2Threads, the streaming ones at kSweep2StreamThreads
__host__ __device__ constexpr int sweep2_threads(int mode) {
  return (mode == S2_MI || mode == S2_GBUF || mode == S2_MSE) ? kSweep2Threads : kSweep2StreamThreads;
}
constexpr int kSweep2Modes = 6;
enum LnccMode { LN_DJ = 0, LN_DU = 1 };  // write dL/dJ; or du and affine partials from the stored slope

// LNCC window sums (windows up to 7) as two kernels: a forward one that stores
// the three g-terms per voxel (12 B/voxel of workspace) and a backward one
// that sums them over the window and runs the epilogue.  FFDP_LNCC_FUSED
// builds the single fused register-history kernel instead (the halo-recompute
// build always uses it).
#ifdef FFDP_LNCC_FUSED
constexpr bool kLnccSplit = false;
#else
constexpr bool kLnccSplit = true;
#endif
#ifndef FFDP_LNCC_SPLIT_MINB
#define FFDP_LNCC_SPLIT_MINB 3
#endif

// Compile-time variant of the LNCC objective path (FFDP_LNCC_RECOMPUTE): the
// window kernel samples J (and, at its output voxels, the slope dJ/dq) from M
// and u on chip instead of reading the J and slope that the histogram sweep
// stores, so the workspace holds nothing per voxel (O(#SMs + B^2)).  The
// default build stores J and the slope (16 B/voxel of workspace).
#ifdef FFDP_LNCC_RECOMPUTE
constexpr bool kLnccRecompute = true;
#else
constexpr bool kLnccRecompute = false;
#endif

// Histogram sweep / forward sampler.
struct Sweep1Args {
  const void* F;
  const void* M;
  const float* u;
  const float* Jin;
  float* Jout;
  float* Gout;                // [N][3] dJ/dq (S1_*WRITEJG)
  unsigned stall_tx;          // tests only: extra bytes armed on ring slot 0 (0 = none)
  unsigned long long* ghist;  // [B*B] fixed-point (kHistFrac) joint histogram
  Geom g;
  BinMap bf, bj;
  int B;
  unsigned nIter;             // CTA iterations of (CTA threads)*kVPT voxels
};

// Gradient sweep: MI table lookups and/or a given dL/dJ, sampler backward.
struct Sweep2Args {
  const void* F;
  const void* M;
  const float* u;
  const float* Jin;   // S2_MI_JBUF, S2_MI_DJ
  const float* gbuf;  // S2_GBUF, S2_GBUF_DJ
  const float* dJdq;  // S2_GBUF_DJ, S2_MI_DJ: [N][3] stored slope of J
  float* du;
  float* dJ;          // S2_MI_JBUF
  const float* T;     // packed MI table (scaled by w_mi * c' / N)
  double* partials;   // [gridDim.x][kPartialStride]
  Geom g;
  BinMap bf, bj;
  int B;
  unsigned nIter;
  float mse_c;        // S2_MSE: g = mse_c (J - F), mse_c = 2 w_mse / N
};

// MI table: normalise the histogram, MI value, packed T = ln P - ln P_F - ln P_J.
struct FinalizeArgs {
  const unsigned long long* ghist;
  float* T;        // gradient table of the linear sweep (polynomial cells for 32 bins)
  float* T2;       // optional: polynomial cells for 64 bins (LNCC-fused gradient)
  double* scalars; // [0 .. BMAX) = MI part of histogram row a
  int B;
  double N;
  double tscale;   // multiplies T (w_mi * (B-5)/(m_hi-m_lo) / N)
};

// LNCC window kernel (J materialised), optional MI gradient and sampler backward.
struct LnccArgs {
  const void* F;
  const float* J;
  const float* dJdq;  // LN_DU: [N][3] stored slope of J
  const void* M;      // halo-recompute build (LN_DU): the moving image, sampled on chip
  const float* u;     //                                and the displacement (NULL: 0)
  float* du;          // LN_DU: [N][3] or NULL (affine partials only)
  float* dJ;          // LN_DJ: [N] dL/dJ or NULL
  float* gbuf;        // split variant: [3][N] g-terms written by the forward kernel
  const float* T;
  double* partials;
  Geom g;          // fixed-grid extents always valid; K and ctr for LN_DU
  BinMap bf, bj;
  int B;
  int R;           // window radius
  float eps;
  float inv_n;     // 1 / window^3
  float gscale;    // -w_lncc / N
  int tilesX, tilesY;  // tile grid (32 x TY columns)
  long long per;       // (column, plane) pairs per CTA
};

// LNCC for windows above kLnccTiledMaxWindow: separable box sums through two
// [5][N] float buffers of the workspace (k_lncc_wide.cu).
constexpr int kLnccTiledMaxWindow = 7;  // tiled register-history kernel (radius <= 3)
struct WideArgs {
  const void* F;
  const float* J;
  const float* dJdq;  // LN_DU: [N][3] stored slope of J
  float* du;          // LN_DU: [N][3] or NULL (affine partials only)
  float* dJ;          // LN_DJ: [N] dL/dJ or NULL
  const float* T;     // MI polynomial cells (B > 0)
  double* partials;   // [grid][kPartialStride]: kPCC from the cc pass, the affine slots from the last pass
  float* bufA;        // [5][N]
  float* bufB;        // [5][N]
  Geom g;             // fixed-grid extents always valid; K and ctr for LN_DU
  BinMap bf, bj;
  int R;              // window radius
  float eps;
  float inv_n;        // 1 / window^3
  float gscale;       // -w_lncc / N
};

// Reduction of per-CTA partials into dA, dt and the loss values.
struct FinishArgs {
  const double* partials;
  int nparts;
  const double* scalars;  // [0 .. mi_rows) = MI parts per histogram row (if MI on)
  int mi_rows;
  float* dA;
  float* dt;
  float* loss;            // NULL or [nloss]
  int nloss;              // 1 (single-term ops), 2 (MSE objective) or 3 (objective)
  double hM[3], xc[3], dx[3];
  double N;
  double w_mi, w_lncc, w_mse;
  int has_mi, has_lncc, has_mse, has_affine;
};

// C-channel sampler (warp composition / image gradient): V is channel-last
// [Dv][Hv][Wv][C] float32; the geometry's moving extents are V's.
struct ChanArgs {
  const float* V;
  const float* u;     // [N][3] or NULL (u = 0)
  const float* gout;  // backward: [N][C]
  float* out;         // forward: [N][C]
  float* du;          // backward: [N][3] or NULL
  float* dV;          // backward: [Dv Hv Wv][C] or NULL (zeroed by the call, then scattered into)
  double* partials;   // backward: [gridDim.x][kPartialStride]
  Geom g;
  float S[9];         // compose: the out / du terms S u and S^T gout
  long long nV;       // Dv Hv Wv C
};

// MSE of a materialised J: per-CTA partial sum (J - F)^2, dJ = c (J - F).
struct MseArgs {
  const void* F;
  const float* J;
  float* dJ;          // or NULL
  double* partials;
  unsigned N;
  float c;            // 2 / N
};

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_zero_u64(unsigned long long* p, int n, cudaStream_t s);
cudaError_t launch_sweep1(int mode, int ft, int mt, int bmax, const Sweep1Args& a, int grid, cudaStream_t s);
cudaError_t launch_sweep2(int mode, int ft, int mt, int bmax, const Sweep2Args& a, int grid, cudaStream_t s);
cudaError_t launch_finalize(int bmax, const FinalizeArgs& a, cudaStream_t s);
cudaError_t launch_lncc(int mode, int ft, int mt, int bmax_or0, const LnccArgs& a, int grid, cudaStream_t s);
cudaError_t launch_lncc_wide(int mode, int ft, int bmax_or0, const WideArgs& a, int grid, cudaStream_t s);
constexpr int kWideCtasPerSm = 8;  // resident 256-thread CTAs per SM of the wide-window passes
cudaError_t launch_finish(const FinishArgs& a, cudaStream_t s);
cudaError_t launch_chan_fwd(int C, int compose, const ChanArgs& a, int grid, cudaStream_t s);
cudaError_t launch_chan_bwd(int C, int compose, const ChanArgs& a, int grid, cudaStream_t s);
cudaError_t launch_zero_f32(float* p, long long n, cudaStream_t s);
cudaError_t launch_mse(int ft, const MseArgs& a, int grid, cudaStream_t s);
int chan_ctas_per_sm(int C, int compose, int bwd);
constexpr int kChanThreads = 256;  // threads per CTA of the channel sampler and the MSE kernel

// Occupancy-derived persistent grid sizes (CTAs per SM), cached per device
// ordinal and kernel variant.  The cache is a table of atomics (zero = not yet
// queried), so host threads may launch concurrently, and each device keeps
// its own counts (GPUs of different kinds in one process).
constexpr int kMaxDevices = 64;
constexpr int kMaxCtasPerSm = 8;
template <int NKEYS>
struct OccCache {
  std::atomic<int> v[kMaxDevices * NKEYS];
  // query() returns resident CTAs per SM (any value; clamped to 1..kMaxCtasPerSm)
  template <class Fn>
  int get(int key, Fn&& query) {
    auto clampv = [](int x) { return x < 1 ? 1 : (x > kMaxCtasPerSm ? kMaxCtasPerSm : x); };
    int dev = 0;
    if (key < 0 || key >= NKEYS || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
      return clampv(query());
    std::atomic<int>& c = v[dev * NKEYS + key];
    int x = c.load(std::memory_order_relaxed);
    if (x == 0) {
      x = clampv(query());
      c.store(x, std::memory_order_relaxed);
    }
    return x;
  }
};
// Test hook: returns and clears the one-shot ring stall request.
unsigned take_test_stall();
// Reads the device error word of the current device (synchronous) and clears it.
cudaError_t take_device_error(unsigned* v);
int sweep1_ctas_per_sm(int mode, int ft, int mt, int bmax);
int sweep2_ctas_per_sm(int mode, int ft, int mt, int bmax);
size_t mi_table_bytes(int bmax);
int lncc_ctas_per_sm(int mode, int ft, int mt, int bmax_or0, int R);

// Timing / launch-count hooks implemented in ffdp_api.cu.
void note_launch_begin(const char* name, cudaStream_t s);
void note_launch_end(cudaStream_t s);

constexpr int kLnccTX = 32;
// LNCC tile height (rows of output voxels per CTA) for window radius <= 2, 3
// and 4, the thread count of the register-history kernel (radius <= 3) and
// the resident CTAs per SM it requests.
#ifndef FFDP_LNCC_TY_SMALL
#define FFDP_LNCC_TY_SMALL 16
#endif
#ifndef FFDP_LNCC_MINB
#define FFDP_LNCC_MINB 2
#endif
#ifndef FFDP_LNCC_THREADS
#define FFDP_LNCC_THREADS 256
#endif
#ifndef FFDP_LNCC_TY_MID
#define FFDP_LNCC_TY_MID 8
#endif
constexpr int kLnccTYSmall = FFDP_LNCC_TY_SMALL;
constexpr int kLnccRHThreads = FFDP_LNCC_THREADS;  // threads per CTA of the register-history LNCC kernel
__host__ __device__ constexpr int lncc_ty(int R) { return R <= 2 ? kLnccTYSmall : (R == 3 ? FFDP_LNCC_TY_MID : 8); }

}  // namespace ffdp
