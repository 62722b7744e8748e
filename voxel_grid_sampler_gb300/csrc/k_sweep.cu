// k_sweep.cu -- voxel-linear sweeps of the fused objective.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration".  Key designs item 1: the composite implicit grid sampler
// I(Ax+t+Su(x)) and its backward (with the affine gradient) run with every
// coordinate in registers.  Key designs item 2: Mattes MI through an implicit
// Parzen window -- histogram entries accumulate per voxel in shared memory and
// the per-voxel partial gradient reads a small table, so no B x N block exists.
//
// Layout of the work: a CTA iteration covers kThreads*kVPT consecutive voxels
// of the flattened [D][H][W] grid; each thread owns kVPT x-consecutive voxels
// so F, J and dJ move as 16-byte vectors and u/du as three 16-byte vectors.
// Grids are persistent (a few CTAs per SM striding over iterations).
#include "ffdp_internal.h"

namespace ffdp {

// ----------------------------------------------------- histogram layout
// Bin (a, b) of the joint histogram has R lane copies: lane l adds into copy
// c = l mod R and visits the four kernel rows rotated by q = (l / R) mod 4.
// Word address = a * SR + b * R + c with row stride SR = BMAX * R + 8
// (8 mod 32), so lanes whose voxels share a base bin always hit distinct words
// in distinct banks, and same-address serialisation cannot occur.
template <int BMAX>
struct HistLayout {
  static constexpr int R = 256 / BMAX;            // 8 copies for 32 bins, 4 for 64
  static constexpr int SR = BMAX * R + 8;          // row stride in words
  static constexpr int WORDS = BMAX * SR;
  // voxels reaching one word per CTA iteration: lanes sharing a copy
  static constexpr int VOX_PER_ITER = kThreads * kVPT / R;
};

// u32 fixed-point counts (kHistFrac fraction bits): one voxel adds at most
// (2/3)^2 to a word, so a CTA flushes its copies to the u64 global histogram
// at least every kFlush<BMAX> iterations.
template <int BMAX>
__host__ __device__ constexpr int flush_every() {
  return (int)(4294967295.0 / (HistLayout<BMAX>::VOX_PER_ITER * (4.0 / 9.0) * kHistOne)) - 1;
}
static_assert(flush_every<32>() >= 16 && flush_every<64>() >= 16, "histogram flush interval");

// fp32 per-thread gradient partials are folded into fp64 every this many iterations.
constexpr int kFoldEvery = 16;

// Fetch the next iteration's F / u group while processing the current one.
#ifndef FFDP_PREFETCH
#define FFDP_PREFETCH 0
#endif
constexpr bool kPrefetch = FFDP_PREFETCH != 0;

__global__ void k_zero_u64(unsigned long long* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0ull;
}

template <int BMAX>
__device__ __forceinline__ void hist_flush(unsigned* hist, unsigned long long* gh, int B) {
  using L = HistLayout<BMAX>;
  __syncthreads();
  for (int i = threadIdx.x; i < B * B; i += kThreads) {
    const int ra = i / B, rb = i - ra * B;
    uint4* w = reinterpret_cast<uint4*>(hist + ra * L::SR + rb * L::R);
    unsigned long long s = 0ull;
#pragma unroll
    for (int k = 0; k < L::R / 4; ++k) {
      const uint4 v = w[k];
      s += (unsigned long long)v.x + v.y + (unsigned long long)v.z + v.w;
      w[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (s) atomicAdd(gh + i, s);
  }
  __syncthreads();
}

// Per-lane constants of the rotated histogram accumulation: polynomial
// coefficients (in t, scaled by 2^kHistFrac) of the cubic B-spline weight of
// kernel row (i + q) mod 4, and that row's word offset.
struct HistLane {
  float c[4][4];
  int rowoff[4];
  int copy;
};

template <int BMAX>
__device__ __forceinline__ void hist_lane_init(HistLane& h) {
  using L = HistLayout<BMAX>;
  // w_j(t) = sum_p W[j][p] t^p for the taps floor(c)-1+j, j = 0..3:
  //   w0 = (1-t)^3/6, w1 = 2/3 - t^2 + t^3/2, w2 = 1/6 + t/2 + t^2/2 - t^3/2, w3 = t^3/6
  const float W[4][4] = {{1.f / 6, -0.5f, 0.5f, -1.f / 6},
                         {2.f / 3, 0.f, -1.f, 0.5f},
                         {1.f / 6, 0.5f, 0.5f, -0.5f},
                         {0.f, 0.f, 0.f, 1.f / 6}};
  const int lane = threadIdx.x & 31;
  const int q = (lane / L::R) & 3;
  h.copy = lane & (L::R - 1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = (i + q) & 3;
#pragma unroll
    for (int p = 0; p < 4; ++p) h.c[i][p] = W[j][p] * kHistOne;
    h.rowoff[i] = j * L::SR;
  }
}

// Parzen contribution of one voxel: beta(a - cF) beta(b - cJ) on the 4x4 bins
// around (cF, cJ), rounded to fixed point with the 1.5*2^23 trick.
template <int BMAX>
__device__ __forceinline__ void hist_add(unsigned* hist, const HistLane& h, const BinMap& bf, const BinMap& bj,
                                         float f, float j) {
  using L = HistLayout<BMAX>;
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float wj[4];
  bspline4(tj, 1.0f, wj);
  unsigned* base = hist + (af - 1) * L::SR + (aj - 1) * L::R + h.copy;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float wf = fmaf(fmaf(fmaf(h.c[i][3], tf, h.c[i][2]), tf, h.c[i][1]), tf, h.c[i][0]);
    unsigned* row = base + h.rowoff[i];
#pragma unroll
    for (int k = 0; k < 4; ++k) atomicAdd(row + k * L::R, __float_as_uint(fmaf(wf, wj[k], kMagic)) - kMagicBits);
  }
}

// ---------------------------------------------------------- MI gradient
// d(w_mi * -MI)/dJ for one voxel = (c'/N) sum_{a,b} T(a,b) beta(a - cF) beta'(b - cJ),
// T = ln P - ln P_F - ln P_J (the +1 and marginal terms of the full chain
// rule cancel by partition of unity).  Zero when J is clamped.
//
// BMAX = 32: per cell (floor cF, floor cJ) the sum is a polynomial of degree
// 3 in tF and 2 in tJ; the MI table kernel stores its 12 coefficients
// (three float4 per cell) and a voxel evaluates it by Horner's rule.
// BMAX = 64: rows of T packed as float2 pairs, 16 taps read directly.
template <int BMAX>
__host__ __device__ constexpr int table_floats() {
  return BMAX == 32 ? BMAX * BMAX * 12 : BMAX * BMAX * 2;
}

template <int BMAX>
__device__ __forceinline__ float mi_grad(const float* tsm, const BinMap& bf, const BinMap& bj, float f,
                                         float j) {
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float s;
  if (BMAX == 32) {
    const float4* c = reinterpret_cast<const float4*>(tsm) + 3 * (af * BMAX + aj);
    const float4 c0 = c[0], c1 = c[1], c2 = c[2];
    // coefficients C[p][r] of tF^p tJ^r: c0 = (C00, C01, C02, C10), c1 = (C11, C12, C20, C21),
    // c2 = (C22, C30, C31, C32)
    const float p0 = fmaf(fmaf(c0.z, tj, c0.y), tj, c0.x);
    const float p1 = fmaf(fmaf(c1.y, tj, c1.x), tj, c0.w);
    const float p2 = fmaf(fmaf(c2.x, tj, c1.w), tj, c1.z);
    const float p3 = fmaf(fmaf(c2.w, tj, c2.z), tj, c2.y);
    s = fmaf(fmaf(fmaf(p3, tf, p2), tf, p1), tf, p0);
  } else {
    float wf[4], d[4];
    bspline4(tf, 1.0f, wf);
    bspline4_deriv(tj, d);
    const float2* t2 = reinterpret_cast<const float2*>(tsm) + (af - 1) * BMAX + (aj - 1);
    s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = t2[i * BMAX], q = t2[i * BMAX + 2];
      s = fmaf(wf[i], fmaf(p.x, d[0], fmaf(p.y, d[1], fmaf(q.x, d[2], q.y * d[3]))), s);
    }
  }
  return (j >= bj.lo && j <= bj.hi) ? s : 0.0f;
}

// ----------------------------------------------------------- group loads
struct Group {
  float f[kVPT], j[kVPT], gb[kVPT], u[3 * kVPT];
};

template <typename FT, bool LOADF, bool LOADU, bool LOADJ, bool LOADG>
__device__ __forceinline__ void load_group(const FT* __restrict__ F, const float* __restrict__ u,
                                           const float* __restrict__ J, const float* __restrict__ gbuf,
                                           unsigned lin0, unsigned nv, Group& G) {
#pragma unroll
  for (int k = 0; k < kVPT; ++k) {
    G.f[k] = 0.f;
    G.j[k] = 0.f;
    G.gb[k] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < 3 * kVPT; ++k) G.u[k] = 0.f;
  if (nv == kVPT) {
    if (LOADF) load4(F + lin0, G.f);
    if (LOADU && u) {
      const float4* up = reinterpret_cast<const float4*>(u + 3ull * lin0);
      const float4 q0 = __ldg(up), q1 = __ldg(up + 1), q2 = __ldg(up + 2);
      G.u[0] = q0.x; G.u[1] = q0.y; G.u[2] = q0.z; G.u[3] = q0.w;
      G.u[4] = q1.x; G.u[5] = q1.y; G.u[6] = q1.z; G.u[7] = q1.w;
      G.u[8] = q2.x; G.u[9] = q2.y; G.u[10] = q2.z; G.u[11] = q2.w;
    }
    if (LOADJ) load4(J + lin0, G.j);
    if (LOADG) load4(gbuf + lin0, G.gb);
  } else {
#pragma unroll
    for (int v = 0; v < kVPT; ++v) {
      if ((unsigned)v < nv) {
        if (LOADF) G.f[v] = load1(F + lin0 + v);
        if (LOADU && u) {
          G.u[3 * v + 0] = __ldg(u + 3ull * (lin0 + v) + 0);
          G.u[3 * v + 1] = __ldg(u + 3ull * (lin0 + v) + 1);
          G.u[3 * v + 2] = __ldg(u + 3ull * (lin0 + v) + 2);
        }
        if (LOADJ) G.j[v] = __ldg(J + lin0 + v);
        if (LOADG) G.gb[v] = __ldg(gbuf + lin0 + v);
      }
    }
  }
}

// Walks the voxels of a 4-voxel group.  Fast path (the group lies in one
// row, always when W % 4 == 0): one fixed-point anchor serves all four.
struct GroupWalk {
  int k[3];
  float f[3];
  int x, y, z;
  bool row;  // whole group in one row
};

__device__ __forceinline__ void walk_begin(const Geom& g, unsigned lin0, GroupWalk& w) {
  lin_to_xyz(g, lin0, w.x, w.y, w.z);
  w.row = g.w4 || (w.x + kVPT <= g.fW);
  anchor_kf(g, w.x, w.y, w.z, w.k, w.f);
}

// Cell of voxel v of the group and its grid index.
__device__ __forceinline__ void walk_cell(const Geom& g, GroupWalk& w, int v, float u0, float u1, float u2,
                                          int b[3], float r[3], int& ix, int& iy, int& iz) {
  if (w.row) {
    cell_v(g, w.k, w.f, (float)v, u0, u1, u2, b, r);
    ix = w.x + v;
    iy = w.y;
    iz = w.z;
  } else {
    if (v > 0) {
      if (++w.x == g.fW) {
        w.x = 0;
        if (++w.y == g.fH) {
          w.y = 0;
          ++w.z;
        }
      }
      anchor_kf(g, w.x, w.y, w.z, w.k, w.f);
    }
    cell_v(g, w.k, w.f, 0.0f, u0, u1, u2, b, r);
    ix = w.x;
    iy = w.y;
    iz = w.z;
  }
}

// Minimum resident CTAs per SM requested from the register allocator.
#ifndef FFDP_SWEEP1_MINB
#define FFDP_SWEEP1_MINB 2
#endif
#ifndef FFDP_SWEEP2_MINB
#define FFDP_SWEEP2_MINB 2
#endif

// ------------------------------------------------------------------ sweep 1
// Sampling (or reading J) plus, per mode, the histogram and/or a J store.
template <typename FT, typename MT, int BMAX, int MODE>
__global__ void __launch_bounds__(kThreads, FFDP_SWEEP1_MINB) k_sweep1(const Sweep1Args a) {
  constexpr bool HIST = MODE != S1_WRITEJ;
  constexpr bool SAMPLE = MODE != S1_HIST_JBUF;
  constexpr bool WRITEJ = (MODE == S1_WRITEJ) || (MODE == S1_HIST_WRITEJ);
  using L = HistLayout<BMAX>;
  extern __shared__ uint4 hist_sm4[];
  unsigned* hist_sm = reinterpret_cast<unsigned*>(hist_sm4);
  const Geom& g = a.g;
  HistLane hl;
  if (HIST) {
    hist_lane_init<BMAX>(hl);
    for (int i = threadIdx.x; i < L::WORDS / 4; i += kThreads) hist_sm4[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  int pending = 0;
  // the F / u group of the next iteration is fetched while this one is processed
  Group Gnext;
  {
    const unsigned l0 = (blockIdx.x * kThreads + threadIdx.x) * kVPT;
    if (kPrefetch && blockIdx.x < a.nIter && l0 < g.N)
      load_group<FT, HIST, SAMPLE, !SAMPLE, false>(F, a.u, a.Jin, nullptr, l0, min(g.N - l0, (unsigned)kVPT), Gnext);
  }
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x) {
    const unsigned lin0 = (it * kThreads + threadIdx.x) * kVPT;
    Group G = Gnext;
    if (kPrefetch) {
      const unsigned itn = it + gridDim.x, ln = (itn * kThreads + threadIdx.x) * kVPT;
      if (itn < a.nIter && ln < g.N)
        load_group<FT, HIST, SAMPLE, !SAMPLE, false>(F, a.u, a.Jin, nullptr, ln, min(g.N - ln, (unsigned)kVPT), Gnext);
    } else if (lin0 < g.N) {
      load_group<FT, HIST, SAMPLE, !SAMPLE, false>(F, a.u, a.Jin, nullptr, lin0, min(g.N - lin0, (unsigned)kVPT), G);
    }
    if (lin0 < g.N) {
      const unsigned nv = min(g.N - lin0, (unsigned)kVPT);
      if (SAMPLE) {
        // all 32 tap loads of the group are issued before any interpolation
        GroupWalk w;
        walk_begin(g, lin0, w);
        float taps[kVPT][8], rr[kVPT][3];
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          int b[3], ix, iy, iz;
          walk_cell(g, w, v, G.u[3 * v], G.u[3 * v + 1], G.u[3 * v + 2], b, rr[v], ix, iy, iz);
          if ((unsigned)v >= nv) b[0] = -2;  // past the end: no loads
          gather8<MT>(M, g, b, taps[v]);
        }
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          float d0, d1, d2;
          G.j[v] = interp8<false>(taps[v], rr[v], d0, d1, d2);
        }
      }
      if (HIST) {
#pragma unroll
        for (int v = 0; v < kVPT; ++v)
          if ((unsigned)v < nv) hist_add<BMAX>(hist_sm, hl, a.bf, a.bj, G.f[v], G.j[v]);
      }
      if (WRITEJ) {
        if (nv == kVPT) {
          *reinterpret_cast<float4*>(a.Jout + lin0) = make_float4(G.j[0], G.j[1], G.j[2], G.j[3]);
        } else {
#pragma unroll
          for (int v = 0; v < kVPT; ++v)
            if ((unsigned)v < nv) a.Jout[lin0 + v] = G.j[v];
        }
      }
    }
    if (HIST && ++pending == flush_every<BMAX>()) {
      hist_flush<BMAX>(hist_sm, a.ghist, a.B);
      pending = 0;
    }
  }
  if (HIST) hist_flush<BMAX>(hist_sm, a.ghist, a.B);
}

// ------------------------------------------------------------ MI finalize
// One CTA: P = H / (N 2^kHistFrac); marginals as row / column sums of the
// joint (equal to the separately defined marginals by partition of unity);
// MI = sum_{P>0} P (ln P - ln P_F - ln P_J); the gradient table of the
// scaled T = tscale (ln P - ln P_F - ln P_J) (0 where P = 0).
template <int BMAX>
__global__ void __launch_bounds__(1024) k_mi_finalize(const FinalizeArgs a) {
  __shared__ double P[BMAX * BMAX];
  __shared__ double PF[BMAX], PJ[BMAX];
  __shared__ double red[32];
  const int B = a.B, nb = B * B, tid = threadIdx.x;
  const double inv = 1.0 / (a.N * (double)kHistOne);
  for (int i = tid; i < nb; i += blockDim.x) P[i] = (double)a.ghist[i] * inv;
  __syncthreads();
  if (tid < B) {
    double s = 0.0;
    for (int b = 0; b < B; ++b) s += P[tid * B + b];
    PF[tid] = s;
  } else if (tid >= 512 && tid - 512 < B) {
    const int b = tid - 512;
    double s = 0.0;
    for (int r = 0; r < B; ++r) s += P[r * B + b];
    PJ[b] = s;
  }
  __syncthreads();
  double mi = 0.0;
  for (int i = tid; i < nb; i += blockDim.x) {
    const int ra = i / B, rb = i - ra * B;
    const double p = P[i];
    double t = 0.0;
    if (p > 0.0) {
      t = log(p) - log(PF[ra]) - log(PJ[rb]);
      mi += p * t;
    }
    P[i] = t * a.tscale;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mi += __shfl_xor_sync(0xffffffffu, mi, o);
  if ((tid & 31) == 0) red[tid >> 5] = mi;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    a.scalars[0] = s;
  }
  auto T = [&](int ra, int rb) -> double { return (ra >= 0 && ra < B && rb >= 0 && rb < B) ? P[ra * B + rb] : 0.0; };
  if (BMAX == 32) {
    // cell (fa, fb): C[p][r] = sum_{i,k} T(fa-1+i, fb-1+k) W[i][p] D[k][r]
    const double W[4][4] = {{1.0 / 6, -0.5, 0.5, -1.0 / 6},
                            {2.0 / 3, 0.0, -1.0, 0.5},
                            {1.0 / 6, 0.5, 0.5, -0.5},
                            {0.0, 0.0, 0.0, 1.0 / 6}};
    // beta'(s) at s = (fb-1+k) - cJ as a polynomial in tJ:
    //   d0 = (1-t)^2/2, d1 = 2t - 1.5t^2, d2 = -1/2 - t + 1.5t^2, d3 = -t^2/2
    const double Dc[4][3] = {{0.5, -1.0, 0.5}, {0.0, 2.0, -1.5}, {-0.5, -1.0, 1.5}, {0.0, 0.0, -0.5}};
    for (int i = tid; i < BMAX * BMAX; i += blockDim.x) {
      const int fa = i / BMAX, fb = i - fa * BMAX;
      double C[4][3] = {};
      for (int ii = 0; ii < 4; ++ii)
        for (int kk = 0; kk < 4; ++kk) {
          const double t = T(fa - 1 + ii, fb - 1 + kk);
          if (t == 0.0) continue;
          for (int p = 0; p < 4; ++p)
            for (int r = 0; r < 3; ++r) C[p][r] += t * W[ii][p] * Dc[kk][r];
        }
      float4* out = reinterpret_cast<float4*>(a.T) + 3 * i;
      out[0] = make_float4((float)C[0][0], (float)C[0][1], (float)C[0][2], (float)C[1][0]);
      out[1] = make_float4((float)C[1][1], (float)C[1][2], (float)C[2][0], (float)C[2][1]);
      out[2] = make_float4((float)C[2][2], (float)C[3][0], (float)C[3][1], (float)C[3][2]);
    }
  } else {
    for (int i = tid; i < BMAX * BMAX; i += blockDim.x) {
      const int ra = i / BMAX, rb = i - ra * BMAX;
      reinterpret_cast<float2*>(a.T)[i] = make_float2((float)T(ra, rb), (float)T(ra, rb + 1));
    }
  }
  // LNCC fusion reads the plain packed table for any bin count
  if (a.T2)
    for (int i = tid; i < BMAX * BMAX; i += blockDim.x) {
      const int ra = i / BMAX, rb = i - ra * BMAX;
      reinterpret_cast<float2*>(a.T2)[i] = make_float2((float)T(ra, rb), (float)T(ra, rb + 1));
    }
}

// ------------------------------------------------------------------ sweep 2
// Per voxel g = dL/dJ (MI table or a given buffer), then either dJ (MI on a
// materialised J) or the sampler backward: du = K^T (g dJ/dq) and the affine
// partial sums, reduced per CTA in fp64.
template <typename FT, typename MT, int BMAX, int MODE>
__global__ void __launch_bounds__(kThreads, FFDP_SWEEP2_MINB) k_sweep2(const Sweep2Args a) {
  constexpr bool MI = MODE != S2_GBUF;
  constexpr bool SAMPLE = MODE != S2_MI_JBUF;
  constexpr bool BWD = MODE != S2_MI_JBUF;
  extern __shared__ float4 tsm4[];
  float* tsm = reinterpret_cast<float*>(tsm4);
  __shared__ double wsum[kThreads / 32][12];
  const Geom& g = a.g;
  if (MI) {
    constexpr int n4 = table_floats<BMAX>() / 4;
    const float4* src = reinterpret_cast<const float4*>(a.T);
    for (int i = threadIdx.x; i < n4; i += kThreads) tsm4[i] = __ldg(src + i);
    __syncthreads();
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  const int warp = threadIdx.x >> 5;
  if (BWD && (threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 12; ++k) wsum[warp][k] = 0.0;
  float acc[12];
#pragma unroll
  for (int k = 0; k < 12; ++k) acc[k] = 0.0f;
  int pending = 0;
  Group Gnext;
  {
    const unsigned l0 = (blockIdx.x * kThreads + threadIdx.x) * kVPT;
    if (kPrefetch && blockIdx.x < a.nIter && l0 < g.N)
      load_group<FT, MI, SAMPLE, !SAMPLE, !MI>(F, a.u, a.Jin, a.gbuf, l0, min(g.N - l0, (unsigned)kVPT), Gnext);
  }
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x) {
    const unsigned lin0 = (it * kThreads + threadIdx.x) * kVPT;
    Group G = Gnext;
    if (kPrefetch) {
      const unsigned itn = it + gridDim.x, ln = (itn * kThreads + threadIdx.x) * kVPT;
      if (itn < a.nIter && ln < g.N)
        load_group<FT, MI, SAMPLE, !SAMPLE, !MI>(F, a.u, a.Jin, a.gbuf, ln, min(g.N - ln, (unsigned)kVPT), Gnext);
    } else if (lin0 < g.N) {
      load_group<FT, MI, SAMPLE, !SAMPLE, !MI>(F, a.u, a.Jin, a.gbuf, lin0, min(g.N - lin0, (unsigned)kVPT), G);
    }
    if (lin0 < g.N) {
      const unsigned nv = min(g.N - lin0, (unsigned)kVPT);
      float out[3 * kVPT];
      if (SAMPLE) {
        // all 32 tap loads of the group are issued before any interpolation
        GroupWalk w;
        walk_begin(g, lin0, w);
        float taps[kVPT][8], rr[kVPT][3];
        int ixv[kVPT], iyv[kVPT], izv[kVPT];
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          int b[3];
          walk_cell(g, w, v, G.u[3 * v], G.u[3 * v + 1], G.u[3 * v + 2], b, rr[v], ixv[v], iyv[v], izv[v]);
          if ((unsigned)v >= nv) b[0] = -2;  // past the end: no loads
          gather8<MT>(M, g, b, taps[v]);
        }
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          out[3 * v + 0] = out[3 * v + 1] = out[3 * v + 2] = 0.0f;
          const int ix = ixv[v], iy = iyv[v], iz = izv[v];
          if ((unsigned)v < nv) {
            float gq0, gq1, gq2;
            const float j = interp8<true>(taps[v], rr[v], gq0, gq1, gq2);
            const float gv = MI ? mi_grad<BMAX>(tsm, a.bf, a.bj, G.f[v], j) : G.gb[v];
            const float e0 = gv * gq0, e1 = gv * gq1, e2 = gv * gq2;
            if (g.k_diag) {
              out[3 * v + 0] = g.K[0] * e0;
              out[3 * v + 1] = g.K[4] * e1;
              out[3 * v + 2] = g.K[8] * e2;
            } else {
              out[3 * v + 0] = fmaf(g.K[0], e0, fmaf(g.K[3], e1, g.K[6] * e2));
              out[3 * v + 1] = fmaf(g.K[1], e0, fmaf(g.K[4], e1, g.K[7] * e2));
              out[3 * v + 2] = fmaf(g.K[2], e0, fmaf(g.K[5], e1, g.K[8] * e2));
            }
            const float cx = (float)ix - g.ctr[0], cy = (float)iy - g.ctr[1], cz = (float)iz - g.ctr[2];
            acc[kPS + 0] += e0;
            acc[kPS + 1] += e1;
            acc[kPS + 2] += e2;
            acc[kPM + 0] = fmaf(e0, cx, acc[kPM + 0]);
            acc[kPM + 1] = fmaf(e0, cy, acc[kPM + 1]);
            acc[kPM + 2] = fmaf(e0, cz, acc[kPM + 2]);
            acc[kPM + 3] = fmaf(e1, cx, acc[kPM + 3]);
            acc[kPM + 4] = fmaf(e1, cy, acc[kPM + 4]);
            acc[kPM + 5] = fmaf(e1, cz, acc[kPM + 5]);
            acc[kPM + 6] = fmaf(e2, cx, acc[kPM + 6]);
            acc[kPM + 7] = fmaf(e2, cy, acc[kPM + 7]);
            acc[kPM + 8] = fmaf(e2, cz, acc[kPM + 8]);
          }
        }
        if (a.du) {
          if (nv == kVPT) {
            float4* dp = reinterpret_cast<float4*>(a.du + 3ull * lin0);
            dp[0] = make_float4(out[0], out[1], out[2], out[3]);
            dp[1] = make_float4(out[4], out[5], out[6], out[7]);
            dp[2] = make_float4(out[8], out[9], out[10], out[11]);
          } else {
#pragma unroll
            for (int v = 0; v < kVPT; ++v)
              if ((unsigned)v < nv) {
                a.du[3ull * (lin0 + v) + 0] = out[3 * v + 0];
                a.du[3ull * (lin0 + v) + 1] = out[3 * v + 1];
                a.du[3ull * (lin0 + v) + 2] = out[3 * v + 2];
              }
          }
        }
      } else {
#pragma unroll
        for (int v = 0; v < kVPT; ++v) out[v] = mi_grad<BMAX>(tsm, a.bf, a.bj, G.f[v], G.j[v]);
        if (nv == kVPT) {
          *reinterpret_cast<float4*>(a.dJ + lin0) = make_float4(out[0], out[1], out[2], out[3]);
        } else {
#pragma unroll
          for (int v = 0; v < kVPT; ++v)
            if ((unsigned)v < nv) a.dJ[lin0 + v] = out[v];
        }
      }
    }
    if (BWD && ++pending == kFoldEvery) {
#pragma unroll
      for (int k = 0; k < 12; ++k) {
        const float s = warp_sum(acc[k]);
        if ((threadIdx.x & 31) == 0) wsum[warp][k] += (double)s;
        acc[k] = 0.0f;
      }
      pending = 0;
    }
  }
  if (BWD) {
#pragma unroll
    for (int k = 0; k < 12; ++k) {
      const float s = warp_sum(acc[k]);
      if ((threadIdx.x & 31) == 0) wsum[warp][k] += (double)s;
    }
    __syncthreads();
    if (threadIdx.x < kPartialStride) {
      double s = 0.0;
      if (threadIdx.x < 12)
        for (int k = 0; k < kThreads / 32; ++k) s += wsum[k][threadIdx.x];
      a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = s;
    }
  }
}

// ------------------------------------------------------------------- finish
// One CTA: fixed-order sum of the per-CTA partials, then
//   dt_r = hM_r s_r,   dA[r][c] = hM_r (xc_c s_r + dx_c m_rc),
// and the loss values.
__global__ void __launch_bounds__(256) k_finish(const FinishArgs a) {
  __shared__ double sm[kPartialStride][17];
  const int c = threadIdx.x & 15, gi = threadIdx.x >> 4;
  double s = 0.0;
  for (int p = gi; p < a.nparts; p += 16) s += a.partials[(size_t)p * kPartialStride + c];
  sm[c][gi] = s;
  __syncthreads();
  if (threadIdx.x < 16) {
    double t = 0.0;
    for (int k = 0; k < 16; ++k) t += sm[threadIdx.x][k];
    sm[threadIdx.x][16] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.has_affine) {
      for (int r = 0; r < 3; ++r) {
        const double sr = sm[kPS + r][16];
        if (a.dt) a.dt[r] = (float)(a.hM[r] * sr);
        if (a.dA)
          for (int cc = 0; cc < 3; ++cc)
            a.dA[r * 3 + cc] = (float)(a.hM[r] * (a.xc[cc] * sr + a.dx[cc] * sm[kPM + r * 3 + cc][16]));
      }
    }
    if (a.loss) {
      const double mi = a.has_mi ? a.scalars[0] : 0.0;
      const double lncc = a.has_lncc ? sm[kPCC][16] / a.N : 0.0;
      if (a.nloss == 3) {
        a.loss[0] = (float)(a.w_mi * (-mi) + a.w_lncc * (-lncc));
        a.loss[1] = (float)(-mi);
        a.loss[2] = (float)(-lncc);
      } else {
        a.loss[0] = (float)(a.has_mi ? -mi : -lncc);
      }
    }
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_zero_u64(unsigned long long* p, int n, cudaStream_t s) {
  note_launch_begin("k_zero_u64", s);
  k_zero_u64<<<(n + 255) / 256 < 64 ? (n + 255) / 256 : 64, 256, 0, s>>>(p, n);
  note_launch_end(s);
  return cudaGetLastError();
}

template <int BMAX, int MODE>
static size_t sweep1_smem() {
  return MODE == S1_WRITEJ ? 0 : (size_t)HistLayout<BMAX>::WORDS * sizeof(unsigned);
}

template <typename FT, typename MT, int BMAX, int MODE>
static cudaError_t run_sweep1(const Sweep1Args& a, int grid, cudaStream_t s, int* occ) {
  auto k = k_sweep1<FT, MT, BMAX, MODE>;
  const size_t smem = sweep1_smem<BMAX, MODE>();
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kThreads, smem);
  note_launch_begin("k_sweep1", s);
  k<<<grid, kThreads, smem, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

static cudaError_t dispatch_sweep1(int mode, int ft, int mt, int bmax, const Sweep1Args& a, int grid,
                                   cudaStream_t s, int* occ) {
  cudaError_t e = cudaErrorInvalidValue;
  FFDP_DT_SWITCH(ft, FT, FFDP_DT_SWITCH(mt, MT, {
    if (bmax == 32) {
      switch (mode) {
        case S1_HIST: e = run_sweep1<FT, MT, 32, S1_HIST>(a, grid, s, occ); break;
        case S1_HIST_WRITEJ: e = run_sweep1<FT, MT, 32, S1_HIST_WRITEJ>(a, grid, s, occ); break;
        case S1_WRITEJ: e = run_sweep1<float, MT, 32, S1_WRITEJ>(a, grid, s, occ); break;
        case S1_HIST_JBUF: e = run_sweep1<FT, float, 32, S1_HIST_JBUF>(a, grid, s, occ); break;
      }
    } else {
      switch (mode) {
        case S1_HIST: e = run_sweep1<FT, MT, 64, S1_HIST>(a, grid, s, occ); break;
        case S1_HIST_WRITEJ: e = run_sweep1<FT, MT, 64, S1_HIST_WRITEJ>(a, grid, s, occ); break;
        case S1_WRITEJ: e = run_sweep1<float, MT, 32, S1_WRITEJ>(a, grid, s, occ); break;
        case S1_HIST_JBUF: e = run_sweep1<FT, float, 64, S1_HIST_JBUF>(a, grid, s, occ); break;
      }
    }
  }));
  return e;
}

cudaError_t launch_sweep1(int mode, int ft, int mt, int bmax, const Sweep1Args& a, int grid, cudaStream_t s) {
  return dispatch_sweep1(mode, ft, mt, bmax, a, grid, s, nullptr);
}

int sweep1_ctas_per_sm(int mode, int ft, int mt, int bmax) {
  static int cache[4][2][2][2] = {};
  int& c = cache[mode][ft][mt][bmax == 64];
  if (c == 0) {
    int occ = 0;
    Sweep1Args dummy{};
    if (dispatch_sweep1(mode, ft, mt, bmax, dummy, 0, 0, &occ) != cudaSuccess || occ < 1) occ = 1;
    c = occ > kMaxCtasPerSm ? kMaxCtasPerSm : occ;
  }
  return c;
}

template <typename FT, typename MT, int BMAX, int MODE>
static cudaError_t run_sweep2(const Sweep2Args& a, int grid, cudaStream_t s, int* occ) {
  auto k = k_sweep2<FT, MT, BMAX, MODE>;
  const size_t smem = MODE == S2_GBUF ? 0 : (size_t)table_floats<BMAX>() * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kThreads, smem);
  note_launch_begin("k_sweep2", s);
  k<<<grid, kThreads, smem, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

static cudaError_t dispatch_sweep2(int mode, int ft, int mt, int bmax, const Sweep2Args& a, int grid,
                                   cudaStream_t s, int* occ) {
  cudaError_t e = cudaErrorInvalidValue;
  FFDP_DT_SWITCH(ft, FT, FFDP_DT_SWITCH(mt, MT, {
    if (bmax == 32) {
      switch (mode) {
        case S2_MI: e = run_sweep2<FT, MT, 32, S2_MI>(a, grid, s, occ); break;
        case S2_GBUF: e = run_sweep2<float, MT, 32, S2_GBUF>(a, grid, s, occ); break;
        case S2_MI_JBUF: e = run_sweep2<FT, float, 32, S2_MI_JBUF>(a, grid, s, occ); break;
      }
    } else {
      switch (mode) {
        case S2_MI: e = run_sweep2<FT, MT, 64, S2_MI>(a, grid, s, occ); break;
        case S2_GBUF: e = run_sweep2<float, MT, 32, S2_GBUF>(a, grid, s, occ); break;
        case S2_MI_JBUF: e = run_sweep2<FT, float, 64, S2_MI_JBUF>(a, grid, s, occ); break;
      }
    }
  }));
  return e;
}

cudaError_t launch_sweep2(int mode, int ft, int mt, int bmax, const Sweep2Args& a, int grid, cudaStream_t s) {
  return dispatch_sweep2(mode, ft, mt, bmax, a, grid, s, nullptr);
}

int sweep2_ctas_per_sm(int mode, int ft, int mt, int bmax) {
  static int cache[3][2][2][2] = {};
  int& c = cache[mode][ft][mt][bmax == 64];
  if (c == 0) {
    int occ = 0;
    Sweep2Args dummy{};
    if (dispatch_sweep2(mode, ft, mt, bmax, dummy, 0, 0, &occ) != cudaSuccess || occ < 1) occ = 1;
    c = occ > kMaxCtasPerSm ? kMaxCtasPerSm : occ;
  }
  return c;
}

cudaError_t launch_finalize(int bmax, const FinalizeArgs& a, cudaStream_t s) {
  note_launch_begin("k_mi_finalize", s);
  if (bmax == 32)
    k_mi_finalize<32><<<1, 1024, 0, s>>>(a);
  else
    k_mi_finalize<64><<<1, 1024, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t launch_finish(const FinishArgs& a, cudaStream_t s) {
  note_launch_begin("k_finish", s);
  k_finish<<<1, 256, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

size_t mi_table_bytes(int bmax) { return (size_t)(bmax == 32 ? table_floats<32>() : table_floats<64>()) * sizeof(float); }

}  // namespace ffdp
