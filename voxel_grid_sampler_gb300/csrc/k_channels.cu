// k_channels.cu -- the composite implicit sampler on a C-channel volume (warp
// composition; with C = 1 also the gradient with respect to the moving
// image) and the MSE similarity of a materialised J.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration".  "Background": L = C(F, M o phi) + R(phi), C one of MSE,
// LNCC or MI, with deformation interpolation and warp composition among the
// memory bottlenecks it profiles.  Key designs item 1: every coordinate of
// I(Ax+t+Su(x)) lives in registers (the identity grid is implicit in
// x_bounds); the backward pass is PyTorch's (gradients to the sampled volume
// and to the coordinates) plus the affine gradient.  Item 5: MSE is a
// per-voxel loss.
//
// Work layout: a persistent grid of kChanThreads-thread CTAs strides over the
// fixed voxels; a warp takes 32 consecutive voxels per step, so its u / gout
// loads and out / du stores cover contiguous spans and the trilinear taps of
// 32 neighbouring points share cache lines of V.  V is channel-last, so the C
// channels of one tap are adjacent (one 16-byte load for C = 4, 8 bytes for
// C = 2).  The image gradient dV is a scatter: every cell row adds gout *
// weight for its two x taps with 16-byte vector reductions (red_pair), which
// L2 resolves; the affine partial sums are kept per thread in fp32 and folded
// into per-warp fp64 sums every kChanFold voxel groups, then per CTA.
#include "ffdp_internal.h"

namespace ffdp {

constexpr int kChanFold = 32;  // voxel groups per warp between fp32 -> fp64 folds

template <int C>
__device__ __forceinline__ void load_tap(const float* __restrict__ V, long long idx, float* v) {
  const float* p = V + idx * C;
  if constexpr (C == 4) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  } else if constexpr (C == 2) {
    const float2 q = __ldg(reinterpret_cast<const float2*>(p));
    v[0] = q.x;
    v[1] = q.y;
  } else {
#pragma unroll
    for (int c = 0; c < C; ++c) v[c] = __ldg(p + c);
  }
}

// Flat tap indices (Dv Hv Wv order) of the 8 corners of cell b, in the
// m[z][y][x] order of interp8; -1 for a corner outside V (reads 0, receives
// nothing).
__device__ __forceinline__ void corner_index(const Geom& g, const int b[3], long long idx[8]) {
  const int bx = b[0], by = b[1], bz = b[2];
  if ((unsigned)bx < (unsigned)(g.mW - 1) && (unsigned)by < (unsigned)(g.mH - 1) &&
      (unsigned)bz < (unsigned)(g.mD - 1)) {
    // interior cell: one base index, fixed corner offsets
    const long long o = ((long long)bz * g.mH + by) * g.mW + bx;
    idx[0] = o;
    idx[1] = o + 1;
    idx[2] = o + g.mW;
    idx[3] = o + g.mW + 1;
    idx[4] = o + g.mHW;
    idx[5] = o + g.mHW + 1;
    idx[6] = o + g.mHW + g.mW;
    idx[7] = o + g.mHW + g.mW + 1;
    return;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int x = bx + (k & 1), y = by + ((k >> 1) & 1), z = bz + (k >> 2);
    const bool in = (unsigned)x < (unsigned)g.mW && (unsigned)y < (unsigned)g.mH && (unsigned)z < (unsigned)g.mD;
    idx[k] = in ? ((long long)z * g.mH + y) * g.mW + x : -1;
  }
}

// The 8 taps of every channel: m[c][k] (k in interp8 order).
template <int C>
__device__ __forceinline__ void gather_c(const float* __restrict__ V, const long long idx[8], float m[C][8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float v[C];
    if (idx[k] >= 0) {
      load_tap<C>(V, idx[k], v);
    } else {
#pragma unroll
      for (int c = 0; c < C; ++c) v[c] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < C; ++c) m[c][k] = v[c];
  }
}

// Adds vals[0 .. 2C) to dV[f0 .. f0 + 2C) (the two x taps of one cell row,
// adjacent in a channel-last volume; a tap outside V has zero vals) with
// vector reductions of kDvChunk floats (8 or 16 bytes) over the aligned
// chunks covering the span, padded with zeros (adding 0 leaves a value
// unchanged).  A chunk that would reach outside dV[0 .. nV) is sent as scalar
// reductions of the span's own elements instead.  The chunk offset
// off = f0 mod kDvChunk selects, for every chunk element, which val (or 0) it
// carries, by compile-time unrolled selects (no dynamically indexed register
// array).
#ifndef FFDP_DV_CHUNK
#define FFDP_DV_CHUNK 4
#endif
constexpr int kDvChunk = FFDP_DV_CHUNK;  // floats per vector reduction of the dV scatter
static_assert(kDvChunk == 2 || kDvChunk == 4, "8- or 16-byte vector reductions");

template <int C>
__device__ __forceinline__ void red_pair(float* __restrict__ dV, long long nV, long long f0, const float vals[2 * C]) {
  constexpr int N = 2 * C, Q = kDvChunk;
  constexpr int NCH = (Q - 1 + N + Q - 1) / Q;  // chunks for the worst offset
  const long long a = f0 & ~(long long)(Q - 1);
  const int off = (int)(f0 - a);
  const int nch = (off + N + Q - 1) / Q;
#pragma unroll
  for (int k = 0; k < NCH; ++k) {
    if (k >= nch) break;
    float v[Q];
#pragma unroll
    for (int j = 0; j < Q; ++j) {
      const int e = Q * k + j;  // element of the chunk run; source val index e - off
      float x = (e < N) ? vals[e] : 0.0f;
#pragma unroll
      for (int o = 1; o < Q; ++o) {
        const float c = (e - o >= 0 && e - o < N) ? vals[e - o] : 0.0f;
        x = off == o ? c : x;
      }
      v[j] = x;
    }
    const long long base = a + Q * k;
    if (base >= 0 && base + Q <= nV) {
      if constexpr (Q == 4)
        atomicAdd(reinterpret_cast<float4*>(dV + base), make_float4(v[0], v[1], v[2], v[3]));
      else
        atomicAdd(reinterpret_cast<float2*>(dV + base), make_float2(v[0], v[1]));
    } else {
#pragma unroll
      for (int j = 0; j < Q; ++j) {
        const int src = Q * k + j - off;
        if (src >= 0 && src < N && base + j >= 0 && base + j < nV) atomicAdd(dV + base + j, v[j]);
      }
    }
  }
}

// Coordinates of fixed voxel lin: indices and the cell of q = G i + g0 + K u.
__device__ __forceinline__ void voxel_cell(const Geom& g, const float* __restrict__ u, unsigned lin, int& ix, int& iy,
                                           int& iz, float uv[3], int b[3], float r[3]) {
  lin_to_xyz(g, lin, ix, iy, iz);
  long long P[3];
  anchor(g, ix, iy, iz, P);
  if (u) {
    uv[0] = __ldg(u + 3ull * lin + 0);
    uv[1] = __ldg(u + 3ull * lin + 1);
    uv[2] = __ldg(u + 3ull * lin + 2);
  } else {
    uv[0] = uv[1] = uv[2] = 0.0f;
  }
  cell_of(g, P, uv[0], uv[1], uv[2], b, r);
}

// out[i][c] = V_c(p_i) (+ (S u_i)_c when COMPOSE).
template <int C, bool COMPOSE>
__global__ void __launch_bounds__(kChanThreads) k_chan_fwd(const ChanArgs a) {
  const Geom& g = a.g;
  const unsigned long long stride = (unsigned long long)gridDim.x * kChanThreads;
  for (unsigned long long l = (unsigned long long)blockIdx.x * kChanThreads + threadIdx.x; l < g.N; l += stride) {
    const unsigned lin = (unsigned)l;
    int ix, iy, iz, b[3];
    float uv[3], r[3];
    voxel_cell(g, a.u, lin, ix, iy, iz, uv, b, r);
    long long idx[8];
    corner_index(g, b, idx);
    float m[C][8];
    gather_c<C>(a.V, idx, m);
    float* o = a.out + (unsigned long long)lin * C;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      float gx, gy, gz;
      float v = interp8<false>(m[c], r, gx, gy, gz);
      if constexpr (COMPOSE) v += fmaf(a.S[c * 3 + 0], uv[0], fmaf(a.S[c * 3 + 1], uv[1], a.S[c * 3 + 2] * uv[2]));
      o[c] = v;
    }
  }
}

// Backward: e = sum_c gout_c dV_c/dq, du = K^T e (+ S^T gout when COMPOSE),
// affine partials of e, and (dV != NULL) dV[tap][c] += gout_c w_tap.  The
// loop runs over warp-uniform groups of 32 voxels, so the periodic warp
// reductions of the partials see every lane.
template <int C, bool COMPOSE>
__global__ void __launch_bounds__(kChanThreads) k_chan_bwd(const ChanArgs a) {
  __shared__ double wsum[kChanThreads / 32][12];
  const Geom& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0)
#pragma unroll
    for (int q = 0; q < 12; ++q) wsum[warp][q] = 0.0;
  float acc[12];
#pragma unroll
  for (int q = 0; q < 12; ++q) acc[q] = 0.0f;
  int pend = 0;
  const unsigned long long stride = (unsigned long long)gridDim.x * kChanThreads;
  for (unsigned long long l0 = (unsigned long long)blockIdx.x * kChanThreads + 32 * warp; l0 < g.N; l0 += stride) {
    if (l0 + lane < g.N) {
      const unsigned lin = (unsigned)(l0 + lane);
      int ix, iy, iz, b[3];
      float uv[3], r[3];
      voxel_cell(g, a.u, lin, ix, iy, iz, uv, b, r);
      long long idx[8];
      corner_index(g, b, idx);
      float go[C];
      load_tap<C>(a.gout, (long long)lin, go);
      float m[C][8];
      gather_c<C>(a.V, idx, m);
      float e0 = 0.0f, e1 = 0.0f, e2 = 0.0f;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        float gx, gy, gz;
        (void)interp8<true>(m[c], r, gx, gy, gz);
        e0 = fmaf(go[c], gx, e0);
        e1 = fmaf(go[c], gy, e1);
        e2 = fmaf(go[c], gz, e2);
      }
      if (a.du) {
        const float* K = g.K;
        float o0 = fmaf(K[0], e0, fmaf(K[3], e1, K[6] * e2));
        float o1 = fmaf(K[1], e0, fmaf(K[4], e1, K[7] * e2));
        float o2 = fmaf(K[2], e0, fmaf(K[5], e1, K[8] * e2));
        if constexpr (COMPOSE) {
          const float* S = a.S;
          o0 += fmaf(S[0], go[0], fmaf(S[3], go[1], S[6] * go[2]));
          o1 += fmaf(S[1], go[0], fmaf(S[4], go[1], S[7] * go[2]));
          o2 += fmaf(S[2], go[0], fmaf(S[5], go[1], S[8] * go[2]));
        }
        float* dp = a.du + 3ull * lin;
        dp[0] = o0;
        dp[1] = o1;
        dp[2] = o2;
      }
      const float e[3] = {e0, e1, e2};
      const float cc[3] = {(float)ix - g.ctr[0], (float)iy - g.ctr[1], (float)iz - g.ctr[2]};
#pragma unroll
      for (int rr = 0; rr < 3; ++rr) {
        acc[kPS + rr] += e[rr];
#pragma unroll
        for (int c = 0; c < 3; ++c) acc[kPM + 3 * rr + c] = fmaf(e[rr], cc[c], acc[kPM + 3 * rr + c]);
      }
      if (a.dV) {
        // per row of the cell, both x taps at once (their 2C floats are adjacent)
        const float wx[2] = {1.0f - r[0], r[0]}, wy[2] = {1.0f - r[1], r[1]}, wz[2] = {1.0f - r[2], r[2]};
#pragma unroll
        for (int row = 0; row < 4; ++row) {
          const int y = b[1] + (row & 1), z = b[2] + (row >> 1);
          if ((unsigned)y >= (unsigned)g.mH || (unsigned)z >= (unsigned)g.mD) continue;
          const float wyz = wy[row & 1] * wz[row >> 1];
          const bool in0 = idx[2 * row] >= 0, in1 = idx[2 * row + 1] >= 0;
          if (!in0 && !in1) continue;
          float vals[2 * C];
#pragma unroll
          for (int c = 0; c < C; ++c) {
            vals[c] = in0 ? go[c] * (wx[0] * wyz) : 0.0f;
            vals[C + c] = in1 ? go[c] * (wx[1] * wyz) : 0.0f;
          }
          const long long f0 = (((long long)z * g.mH + y) * g.mW + b[0]) * C;
          red_pair<C>(a.dV, a.nV, f0, vals);
        }
      }
    }
    if (++pend == kChanFold) {
#pragma unroll
      for (int q = 0; q < 12; ++q) {
        const float s = warp_sum(acc[q]);
        if (lane == 0) wsum[warp][q] += (double)s;
        acc[q] = 0.0f;
      }
      pend = 0;
    }
  }
#pragma unroll
  for (int q = 0; q < 12; ++q) {
    const float s = warp_sum(acc[q]);
    if (lane == 0) wsum[warp][q] += (double)s;
  }
  __syncthreads();
  if (threadIdx.x < kPartialStride) {
    double s = 0.0;
    if (threadIdx.x < 12)
      for (int w = 0; w < kChanThreads / 32; ++w) s += wsum[w][threadIdx.x];
    a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = s;
  }
}

// p[0 .. n) = 0 (p 16-byte aligned).
__global__ void __launch_bounds__(256) k_zero_f32(float* p, long long n) {
  const long long n4 = n / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float4* p4 = reinterpret_cast<float4*>(p);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) p[4 * n4 + threadIdx.x] = 0.0f;
}

// Four fixed-image values starting at element 4 i (16-byte / 8-byte aligned).
__device__ __forceinline__ void load4(const float* __restrict__ F, unsigned long long i, float f[4]) {
  const float4 q = __ldg(reinterpret_cast<const float4*>(F) + i);
  f[0] = q.x;
  f[1] = q.y;
  f[2] = q.z;
  f[3] = q.w;
}
__device__ __forceinline__ void load4(const __half* __restrict__ F, unsigned long long i, float f[4]) {
  const uint2 q = __ldg(reinterpret_cast<const uint2*>(F) + i);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// MSE of a materialised J: per-CTA sum (J - F)^2 into record slot kPSE and
// dJ = c (J - F), four voxels per thread step (16-byte vectors).
template <typename FT>
__global__ void __launch_bounds__(kChanThreads) k_mse(const MseArgs a) {
  __shared__ double red[kChanThreads / 32];
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const unsigned long long n4 = a.N / 4;
  const unsigned long long stride = (unsigned long long)gridDim.x * kChanThreads;
  float acc = 0.0f;
  double dacc = 0.0;
  int pend = 0;
  for (unsigned long long i = (unsigned long long)blockIdx.x * kChanThreads + threadIdx.x; i < n4; i += stride) {
    float f[4];
    load4(F, i, f);
    const float4 j = __ldg(reinterpret_cast<const float4*>(a.J) + i);
    const float d0 = j.x - f[0], d1 = j.y - f[1], d2 = j.z - f[2], d3 = j.w - f[3];
    acc = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, acc))));
    if (a.dJ) reinterpret_cast<float4*>(a.dJ)[i] = make_float4(a.c * d0, a.c * d1, a.c * d2, a.c * d3);
    if (++pend == kChanFold) {
      dacc += (double)acc;
      acc = 0.0f;
      pend = 0;
    }
  }
  // the last N mod 4 voxels
  if (blockIdx.x == 0 && threadIdx.x < (a.N & 3u)) {
    const unsigned k = 4u * (unsigned)n4 + threadIdx.x;
    const float d = __ldg(a.J + k) - load1(F + k);
    acc = fmaf(d, d, acc);
    if (a.dJ) a.dJ[k] = a.c * d;
  }
  double v = dacc + (double)acc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < kPartialStride) {
    double s = 0.0;
    if (threadIdx.x == kPSE)
      for (int w = 0; w < kChanThreads / 32; ++w) s += red[w];
    a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = s;
  }
}

// ---------------------------------------------------------------- launchers
#define FFDP_CHAN_SWITCH(C, COMPOSE, ...)                                  \
  do {                                                                     \
    if ((COMPOSE)) {                                                       \
      constexpr int kC = 3;                                                \
      constexpr bool kComp = true;                                         \
      __VA_ARGS__;                                                         \
    } else if ((C) == 1) {                                                 \
      constexpr int kC = 1;                                                \
      constexpr bool kComp = false;                                        \
      __VA_ARGS__;                                                         \
    } else if ((C) == 2) {                                                 \
      constexpr int kC = 2;                                                \
      constexpr bool kComp = false;                                        \
      __VA_ARGS__;                                                         \
    } else if ((C) == 3) {                                                 \
      constexpr int kC = 3;                                                \
      constexpr bool kComp = false;                                        \
      __VA_ARGS__;                                                         \
    } else {                                                               \
      constexpr int kC = 4;                                                \
      constexpr bool kComp = false;                                        \
      __VA_ARGS__;                                                         \
    }                                                                      \
  } while (0)

template <int C, bool COMPOSE>
static void run_chan_fwd(const ChanArgs& a, int grid, cudaStream_t s) {
  k_chan_fwd<C, COMPOSE><<<grid, kChanThreads, 0, s>>>(a);
}
template <int C, bool COMPOSE>
static void run_chan_bwd(const ChanArgs& a, int grid, cudaStream_t s) {
  k_chan_bwd<C, COMPOSE><<<grid, kChanThreads, 0, s>>>(a);
}

cudaError_t launch_chan_fwd(int C, int compose, const ChanArgs& a, int grid, cudaStream_t s) {
  note_launch_begin("k_chan_fwd", s);
  FFDP_CHAN_SWITCH(C, compose, run_chan_fwd<kC, kComp>(a, grid, s));
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t launch_chan_bwd(int C, int compose, const ChanArgs& a, int grid, cudaStream_t s) {
  note_launch_begin("k_chan_bwd", s);
  FFDP_CHAN_SWITCH(C, compose, run_chan_bwd<kC, kComp>(a, grid, s));
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t launch_zero_f32(float* p, long long n, cudaStream_t s) {
  long long blocks = (n / 4 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 4096) blocks = 4096;
  note_launch_begin("k_zero_f32", s);
  k_zero_f32<<<(int)blocks, 256, 0, s>>>(p, n);
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t launch_mse(int ft, const MseArgs& a, int grid, cudaStream_t s) {
  note_launch_begin("k_mse", s);
  if (ft == 0)
    k_mse<float><<<grid, kChanThreads, 0, s>>>(a);
  else
    k_mse<__half><<<grid, kChanThreads, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

// Resident CTAs per SM of the channel kernels (bwd: backward; C = 0: k_mse).
int chan_ctas_per_sm(int C, int compose, int bwd) {
  static OccCache<2 * 5 * 2> cache;
  return cache.get(((bwd ? 1 : 0) * 5 + C) * 2 + (compose ? 1 : 0), [&] {
    int occ = 0;
    cudaError_t e = cudaErrorInvalidValue;
    if (C == 0) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_mse<float>, kChanThreads, 0);
    } else if (bwd) {
      FFDP_CHAN_SWITCH(C, compose, e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_chan_bwd<kC, kComp>, kChanThreads, 0));
    } else {
      FFDP_CHAN_SWITCH(C, compose, e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_chan_fwd<kC, kComp>, kChanThreads, 0));
    }
    return e == cudaSuccess ? occ : 1;
  });
}

}  // namespace ffdp
