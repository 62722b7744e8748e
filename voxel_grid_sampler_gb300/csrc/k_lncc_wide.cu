// k_lncc_wide.cu -- LNCC for windows wider than the tiled kernel keeps on chip
// (w > kLnccTiledMaxWindow).
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration", Key designs item 2 (LNCC from the window sums of I, J, I^2,
// J^2, IJ, and its gradient through the same window sums).  The definitions
// are those of the tiled kernels (zero padding, window w = 2R + 1, n = w^3):
//   cross = S_FJ - S_F S_J / n,  vF = S_FF - S_F^2 / n,  vJ = S_JJ - S_J^2 / n
//   (variances clamped at 0), cc = cross^2 / (vF vJ + eps),
//   D = vF vJ + eps, A1 = 2 cross / D, A2 = cross^2 vF / D^2, s = -w_lncc / N:
//   g_FJ = s A1,  g_JJ = -s A2,  g_J = s (2 A2 S_J - A1 S_F) / n,
//   dJ_m = sum_{k in window(m)} g_J(k) + 2 J_m g_JJ(k) + F_m g_FJ(k).
//
// A window of w^3 voxels with a 2R halo around a 32-wide tile no longer fits
// the register history of the tiled kernel, so the window
// sums run as separable box sums, one grid-stride pass per axis, through two
// [5][N] float buffers A and B of the workspace:
//   1. x sums of J, F, J^2, F^2, FJ                     J, F -> A[0..4]
//   2. y sums                                           A    -> B[0..4]
//   3. z sums, cc (per-CTA partials), g_J, g_JJ, g_FJ    B    -> A[0..2]
//   4. x sums of the three g-terms                      A    -> B[0..2]
//   5. y sums                                           B    -> A[0..2]
//   6. z sums, dJ (+ the MI term from the polynomial cells), then dJ stored
//      or the sampler backward from the stored slope: du = K^T (g dJ/dq) and
//      the affine moments, per-CTA fp64 partials.
// The x sums add the terms inside the grid directly (min(w, extent) loads per
// channel and output, the w-fold reuse of an input served by L1).  The y and z
// sums run along lines: a thread owns 16 consecutive outputs of a line, sums
// the first window directly and slides it along the rest, so the drift of the
// running sum is bounded by 16 steps and each input is loaded about twice.  A
// warp's lanes hold 32 consecutive x, so every load is coalesced.
#include "ffdp_internal.h"
#include "ffdp_lncc.cuh"

namespace ffdp {

constexpr int kWideThreads = 256;

// Window range [lo, hi] along AXIS (0 = x, 1 = y, 2 = z) of voxel lin, clipped
// to the grid, and the element stride of that axis.
template <int AXIS>
__device__ __forceinline__ void axis_window(const Geom& g, unsigned lin, int R, int& lo, int& hi, long long& st) {
  int ix, iy, iz;
  lin_to_xyz(g, lin, ix, iy, iz);
  const int c = AXIS == 0 ? ix : (AXIS == 1 ? iy : iz);
  const int n = AXIS == 0 ? g.fW : (AXIS == 1 ? g.fH : g.fD);
  lo = c - R < 0 ? -c : -R;
  hi = c + R > n - 1 ? n - 1 - c : R;
  st = AXIS == 0 ? 1ll : (AXIS == 1 ? (long long)g.fW : (long long)g.fW * g.fH);
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// pass 1: x sums of the five products of (J, F)
template <typename FT>
__global__ void __launch_bounds__(kWideThreads) k_wide_prod_x(const WideArgs a) {
  const Geom& g = a.g;
  const size_t N = g.N;
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  for (size_t lin = (size_t)blockIdx.x * kWideThreads + threadIdx.x; lin < N; lin += (size_t)gridDim.x * kWideThreads) {
    int lo, hi;
    long long st;
    axis_window<0>(g, (unsigned)lin, a.R, lo, hi, st);
    float sJ = 0.f, sF = 0.f, sJJ = 0.f, sFF = 0.f, sFJ = 0.f;
    for (int k = lo; k <= hi; ++k) {
      const float j = __ldg(a.J + lin + k), f = load1(F + lin + k);
      sJ += j;
      sF += f;
      sJJ = fmaf(j, j, sJJ);
      sFF = fmaf(f, f, sFF);
      sFJ = fmaf(f, j, sFJ);
    }
    a.bufA[lin] = sJ;
    a.bufA[N + lin] = sF;
    a.bufA[2 * N + lin] = sJJ;
    a.bufA[3 * N + lin] = sFF;
    a.bufA[4 * N + lin] = sFJ;
  }
}

// Runs along y or z: a thread owns kRun consecutive outputs of one grid line
// along AXIS and slides its window sums along them (one add and one subtract
// per output after the first full sum), so a y or z pass loads each input
// about twice instead of w times.  Lanes of a warp hold consecutive x, so every
// load is coalesced.
constexpr int kRun = 16;

struct Run {
  size_t base;    // linear index of the run's first output
  long long st;   // element stride along the axis
  int p0, n;      // axis coordinate of the first output, outputs in the run
  int ext;        // grid extent along the axis
  int x, y, z;    // coordinates of the first output
};

// Decodes work item `item` (x fastest) into the run it owns; false past the
// last run.
template <int AXIS>
__device__ __forceinline__ bool run_of(const Geom& g, size_t item, Run& r) {
  const int W = g.fW, H = g.fH, D = g.fD;
  r.ext = AXIS == 1 ? H : D;
  const int nch = (r.ext + kRun - 1) / kRun;
  r.x = (int)(item % (size_t)W);
  const size_t rest = item / (size_t)W;
  int c;
  if (AXIS == 1) {
    c = (int)(rest % (size_t)nch);
    r.z = (int)(rest / (size_t)nch);
    if (r.z >= D) return false;
    r.y = c * kRun;
  } else {
    r.y = (int)(rest % (size_t)H);
    c = (int)(rest / (size_t)H);
    if (c >= nch) return false;
    r.z = c * kRun;
  }
  r.p0 = c * kRun;
  r.n = min(kRun, r.ext - r.p0);
  r.st = AXIS == 1 ? (long long)W : (long long)W * H;
  r.base = ((size_t)r.z * H + r.y) * W + r.x;
  return true;
}

template <int AXIS>
__device__ __forceinline__ size_t runs_total(const Geom& g) {
  const int ext = AXIS == 1 ? g.fH : g.fD;
  const size_t nch = (size_t)((ext + kRun - 1) / kRun);
  return AXIS == 1 ? (size_t)g.fW * nch * g.fD : (size_t)g.fW * g.fH * nch;
}

// Window sums of C channels ([C][N], channel stride N) over the run's
// outputs: emit(i, s) receives output i's sums.  The first output's window is
// summed directly; each next one adds the entering and drops the leaving
// input (zero padding outside the grid).
template <int C, class Emit>
__device__ __forceinline__ void run_sums(const float* __restrict__ in, size_t N, const Run& r, int R, Emit&& emit) {
  float s[C];
#pragma unroll
  for (int c = 0; c < C; ++c) s[c] = 0.f;
  {
    const int lo = r.p0 - R < 0 ? -r.p0 : -R;
    const int hi = r.p0 + R > r.ext - 1 ? r.ext - 1 - r.p0 : R;
    const float* p = in + r.base + (long long)lo * r.st;
    for (int k = lo; k <= hi; ++k, p += r.st) {
#pragma unroll
      for (int c = 0; c < C; ++c) s[c] += __ldg(p + c * N);
    }
  }
  emit(0, s);
  for (int i = 1; i < r.n; ++i) {
    const int pin = r.p0 + i + R, pout = r.p0 + i - R - 1;
    if (pin < r.ext) {
      const float* p = in + r.base + (long long)(i + R) * r.st;
#pragma unroll
      for (int c = 0; c < C; ++c) s[c] += __ldg(p + c * N);
    }
    if (pout >= 0) {
      const float* p = in + r.base + (long long)(i - R - 1) * r.st;
#pragma unroll
      for (int c = 0; c < C; ++c) s[c] -= __ldg(p + c * N);
    }
    emit(i, s);
  }
}

// pass 4: window sums of C channels along x, direct (the w inputs of
// neighbouring lanes overlap and come from L1)
template <int C>
__global__ void __launch_bounds__(kWideThreads) k_wide_box_x(const float* __restrict__ in, float* __restrict__ out,
                                                             const Geom g, int R) {
  const size_t N = g.N;
  for (size_t lin = (size_t)blockIdx.x * kWideThreads + threadIdx.x; lin < N; lin += (size_t)gridDim.x * kWideThreads) {
    int lo, hi;
    long long st;
    axis_window<0>(g, (unsigned)lin, R, lo, hi, st);
    float s[C];
#pragma unroll
    for (int c = 0; c < C; ++c) s[c] = 0.f;
    const float* p = in + lin + lo;
    for (int k = lo; k <= hi; ++k, ++p) {
#pragma unroll
      for (int c = 0; c < C; ++c) s[c] += __ldg(p + c * N);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) out[c * N + lin] = s[c];
  }
}

// passes 2, 5: window sums of C channels along y, by runs
template <int C>
__global__ void __launch_bounds__(kWideThreads) k_wide_box_y(const float* __restrict__ in, float* __restrict__ out,
                                                             const Geom g, int R) {
  const size_t N = g.N, total = runs_total<1>(g);
  for (size_t item = (size_t)blockIdx.x * kWideThreads + threadIdx.x; item < total;
       item += (size_t)gridDim.x * kWideThreads) {
    Run r;
    if (!run_of<1>(g, item, r)) continue;
    run_sums<C>(in, N, r, R, [&](int i, const float* s) {
      const size_t o = r.base + (size_t)i * r.st;
#pragma unroll
      for (int c = 0; c < C; ++c) out[c * N + o] = s[c];
    });
  }
}

// pass 3: z sums of the five channels by runs, cc and the three g-terms
__global__ void __launch_bounds__(kWideThreads) k_wide_cc(const WideArgs a) {
  __shared__ double red[kWideThreads / 32];
  const Geom& g = a.g;
  const size_t N = g.N, total = runs_total<2>(g);
  const float inv_n = a.inv_n, eps = a.eps, gs = a.gscale;
  double cc_d = 0.0;
  for (size_t item = (size_t)blockIdx.x * kWideThreads + threadIdx.x; item < total;
       item += (size_t)gridDim.x * kWideThreads) {
    Run r;
    if (!run_of<2>(g, item, r)) continue;
    float cc_f = 0.0f;  // at most kRun terms, then folded
    run_sums<5>(a.bufB, N, r, a.R, [&](int i, const float* s) {
      const size_t o = r.base + (size_t)i * r.st;
      const float SJ = s[0], SF = s[1];
      const float vJ = fmaxf(fmaf(SJ * SJ, -inv_n, s[2]), 0.0f);
      const float vF = fmaxf(fmaf(SF * SF, -inv_n, s[3]), 0.0f);
      const float cross = fmaf(-SJ * SF, inv_n, s[4]);
      const float rD = rcp_approx(fmaf(vJ, vF, eps));
      const float A1 = 2.0f * cross * rD;
      const float cc = cross * cross * rD;
      const float A2 = cc * vF * rD;
      a.bufA[o] = gs * (2.0f * A2 * SJ - A1 * SF) * inv_n;
      a.bufA[N + o] = -gs * A2;
      a.bufA[2 * N + o] = gs * A1;
      cc_f += cc;
    });
    cc_d += (double)cc_f;
  }
  cc_d = warp_sum_d(cc_d);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cc_d;
  __syncthreads();
  // the whole record: cc, zeros elsewhere (the last pass adds the affine
  // slots in the objective)
  if (threadIdx.x < kPartialStride) {
    double t = 0.0;
    if (threadIdx.x == kPCC)
      for (int w = 0; w < kWideThreads / 32; ++w) t += red[w];
    a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = t;
  }
}

// pass 6: z sums of the g-terms by runs, dJ, and dJ or the sampler backward
template <typename FT, int BMAX, bool DU>
__global__ void __launch_bounds__(kWideThreads) k_wide_fin(const WideArgs a) {
  constexpr bool MI = BMAX != 0;
  // affine moments e_r and e_r (i_c - ctr_c): fp32 over one run, then added
  // to the thread's fp64 slots here (slot kPS + r, kPM + 3 r + c), which keeps
  // them out of the registers of the run loop
  __shared__ double acc[DU ? 12 : 1][kWideThreads];
  const Geom& g = a.g;
  const size_t N = g.N, total = runs_total<2>(g);
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const int tid = threadIdx.x;
  if constexpr (DU)
    for (int c = 0; c < 12; ++c) acc[c][tid] = 0.0;
  for (size_t item = (size_t)blockIdx.x * kWideThreads + threadIdx.x; item < total;
       item += (size_t)gridDim.x * kWideThreads) {
    Run r;
    if (!run_of<2>(g, item, r)) continue;
    float S[3] = {0.f, 0.f, 0.f}, Mo[3][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}};
    const float cx = (float)r.x - g.ctr[0], cy = (float)r.y - g.ctr[1];
    run_sums<3>(a.bufA, N, r, a.R, [&](int i, const float* s) {
      const size_t o = r.base + (size_t)i * r.st;
      const float jv = __ldg(a.J + o), fv = load1(F + o);
      float gv = fmaf(fv, s[2], fmaf(2.0f * jv, s[1], s[0]));
      if (MI) gv += mi_grad_ln<(MI ? BMAX : 32)>(a.T, a.bf, a.bj, fv, jv);
      if constexpr (!DU) {
        if (a.dJ) a.dJ[o] = gv;
      } else {
        const float e[3] = {gv * __ldg(a.dJdq + 3 * o), gv * __ldg(a.dJdq + 3 * o + 1),
                            gv * __ldg(a.dJdq + 3 * o + 2)};
        if (a.du) {
          const float* K = g.K;
          float* d = a.du + 3 * o;
          if (g.k_diag) {
            d[0] = K[0] * e[0];
            d[1] = K[4] * e[1];
            d[2] = K[8] * e[2];
          } else {
            d[0] = fmaf(K[0], e[0], fmaf(K[3], e[1], K[6] * e[2]));
            d[1] = fmaf(K[1], e[0], fmaf(K[4], e[1], K[7] * e[2]));
            d[2] = fmaf(K[2], e[0], fmaf(K[5], e[1], K[8] * e[2]));
          }
        }
        const float cz = (float)(r.z + i) - g.ctr[2];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          S[q] += e[q];
          Mo[q][2] = fmaf(e[q], cz, Mo[q][2]);
        }
      }
    });
    if constexpr (DU) {
      // the run's x and y are fixed: their moments follow from the sums
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        acc[kPS + q][tid] += (double)S[q];
        acc[kPM + 3 * q][tid] += (double)(S[q] * cx);
        acc[kPM + 3 * q + 1][tid] += (double)(S[q] * cy);
        acc[kPM + 3 * q + 2][tid] += (double)Mo[q][2];
      }
    }
  }
  if constexpr (DU) {
    // each warp sums a slot over the CTA's threads (warp w takes slots w, w + 8)
    __syncthreads();
    const int lane = tid & 31, wid = tid >> 5;
    for (int c = wid; c < 12; c += kWideThreads / 32) {
      double t = 0.0;
      for (int k = lane; k < kWideThreads; k += 32) t += acc[c][k];
      t = warp_sum_d(t);
      if (lane == 0) a.partials[(size_t)blockIdx.x * kPartialStride + c] = t;
    }
  }
}

namespace {

template <typename FT, int BMAX, bool DU>
cudaError_t run_wide(const WideArgs& a, int grid, cudaStream_t s) {
  const Geom& g = a.g;
  note_launch_begin("k_wide_prod_x", s);
  k_wide_prod_x<FT><<<grid, kWideThreads, 0, s>>>(a);
  note_launch_end(s);
  note_launch_begin("k_wide_y", s);
  k_wide_box_y<5><<<grid, kWideThreads, 0, s>>>(a.bufA, a.bufB, g, a.R);
  note_launch_end(s);
  note_launch_begin("k_wide_cc", s);
  k_wide_cc<<<grid, kWideThreads, 0, s>>>(a);
  note_launch_end(s);
  note_launch_begin("k_wide_gx", s);
  k_wide_box_x<3><<<grid, kWideThreads, 0, s>>>(a.bufA, a.bufB, g, a.R);
  note_launch_end(s);
  note_launch_begin("k_wide_gy", s);
  k_wide_box_y<3><<<grid, kWideThreads, 0, s>>>(a.bufB, a.bufA, g, a.R);
  note_launch_end(s);
  note_launch_begin("k_wide_fin", s);
  k_wide_fin<FT, BMAX, DU><<<grid, kWideThreads, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

template <typename FT, int BMAX>
cudaError_t run_wide_mode(int mode, const WideArgs& a, int grid, cudaStream_t s) {
  return mode == LN_DU ? run_wide<FT, BMAX, true>(a, grid, s) : run_wide<FT, BMAX, false>(a, grid, s);
}

}  // namespace

cudaError_t launch_lncc_wide(int mode, int ft, int bmax, const WideArgs& a, int grid, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  FFDP_DT_SWITCH(ft, FT, {
    if (bmax == 0)
      e = run_wide_mode<FT, 0>(mode, a, grid, s);
    else if (bmax == 32)
      e = run_wide_mode<FT, 32>(mode, a, grid, s);
    else
      e = run_wide_mode<FT, 64>(mode, a, grid, s);
  });
  return e;
}

}  // namespace ffdp
