// k_sweep.cu -- voxel-linear sweeps of the fused objective.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration".  Key designs item 1: the composite implicit grid sampler
// I(Ax+t+Su(x)) and its backward (with the affine gradient) run with every
// coordinate in registers.  Key designs item 2: Mattes MI through an implicit
// Parzen window -- histogram entries accumulate per voxel in shared memory and
// the per-voxel partial gradient reads a B x B table, so no B x N block exists.
//
// Layout of the work: a CTA iteration covers kThreads*kVPT consecutive voxels
// of the flattened [D][H][W] grid; each thread owns kVPT x-consecutive voxels
// so F, J and dJ move as 16-byte vectors and u/du as three 16-byte vectors.
// Grids are persistent (a few CTAs per SM striding over iterations).
#include "ffdp_internal.h"

namespace ffdp {

// Histogram counts are u32 fixed point with kHistFrac fraction bits.  One
// voxel adds at most (2/3)^2 to a bin, so a CTA may accumulate this many
// iterations before its shared copy must be flushed to the u64 global
// histogram without overflow.
constexpr int kFlushEvery = 8;
static_assert((double)kFlushEvery * kThreads * kVPT * (4.0 / 9.0) * kHistOne < 4294967296.0,
              "histogram flush interval overflows u32");
// fp32 per-thread gradient partials are folded into fp64 every this many iterations.
constexpr int kFoldEvery = 16;

__global__ void k_zero_u64(unsigned long long* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0ull;
}

template <int BMAX>
__device__ __forceinline__ void hist_flush(unsigned* hist, unsigned long long* gh, int B) {
  constexpr int STRIDE = BMAX + 8;
  __syncthreads();
  for (int i = threadIdx.x; i < B * STRIDE; i += kThreads) {
    const unsigned v = hist[i];
    if (v) {
      const int ra = i / STRIDE;
      atomicAdd(gh + ra * B + (i - ra * STRIDE), (unsigned long long)v);
      hist[i] = 0u;
    }
  }
  __syncthreads();
}

// Parzen contribution of one voxel: beta(a - cF) beta(b - cJ) on the 4x4 bins
// around (cF, cJ), rounded to fixed point with the 1.5*2^23 trick.  Rows are
// padded to BMAX+8 words so the four rows of a voxel hit distinct banks;
// lanes adding to one address are combined by the shared-memory atomic unit.
template <int BMAX>
__device__ __forceinline__ void hist_add(unsigned* hist, const BinMap& bf, const BinMap& bj, float f,
                                         float j) {
  constexpr int STRIDE = BMAX + 8;
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float wf[4], wj[4];
  bspline4(tf, kHistOne, wf);
  bspline4(tj, 1.0f, wj);
  unsigned* h = hist + (af - 1) * STRIDE + (aj - 1);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      atomicAdd(h + i * STRIDE + k, __float_as_uint(fmaf(wf[i], wj[k], kMagic)) - kMagicBits);
}

// d(w_mi * -MI)/dJ for one voxel: sum_{a,b} T'(a,b) beta(a - cF) beta'(b - cJ),
// T' = w_mi * c'/N * (ln P - ln P_F - ln P_J); zero when J is clamped.
template <int BMAX>
__device__ __forceinline__ float mi_grad(const float* tsm, const BinMap& bf, const BinMap& bj, float f,
                                         float j) {
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float wf[4], d[4];
  bspline4(tf, 1.0f, wf);
  bspline4_deriv(tj, d);
  float s = 0.0f;
  if (BMAX == 32) {
    const float4* t4 = reinterpret_cast<const float4*>(tsm) + (af - 1) * BMAX + (aj - 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = t4[i * BMAX];
      s = fmaf(wf[i], fmaf(t.x, d[0], fmaf(t.y, d[1], fmaf(t.z, d[2], t.w * d[3]))), s);
    }
  } else {
    const float2* t2 = reinterpret_cast<const float2*>(tsm) + (af - 1) * BMAX + (aj - 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = t2[i * BMAX], q = t2[i * BMAX + 2];
      s = fmaf(wf[i], fmaf(p.x, d[0], fmaf(p.y, d[1], fmaf(q.x, d[2], q.y * d[3]))), s);
    }
  }
  return (j >= bj.lo && j <= bj.hi) ? s : 0.0f;
}

template <int BMAX>
__host__ __device__ constexpr int table_floats() {
  return BMAX == 32 ? BMAX * BMAX * 4 : BMAX * BMAX * 2;
}

// ------------------------------------------------------------------ sweep 1
// Sampling (or reading J) plus, per mode, the histogram and/or a J store.
template <typename FT, typename MT, int BMAX, int MODE>
__global__ void __launch_bounds__(kThreads) k_sweep1(const Sweep1Args a) {
  constexpr bool HIST = MODE != S1_WRITEJ;
  constexpr bool SAMPLE = MODE != S1_HIST_JBUF;
  constexpr bool WRITEJ = (MODE == S1_WRITEJ) || (MODE == S1_HIST_WRITEJ);
  constexpr int STRIDE = BMAX + 8;
  extern __shared__ unsigned hist_sm[];
  const Geom& g = a.g;
  if (HIST) {
    for (int i = threadIdx.x; i < BMAX * STRIDE; i += kThreads) hist_sm[i] = 0u;
    __syncthreads();
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  int pending = 0;
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x) {
    const unsigned lin0 = (it * kThreads + threadIdx.x) * kVPT;
    if (lin0 < g.N) {
      const unsigned nv = min(g.N - lin0, (unsigned)kVPT);
      float fv[kVPT] = {0.f, 0.f, 0.f, 0.f}, jv[kVPT] = {0.f, 0.f, 0.f, 0.f}, uv[3 * kVPT];
#pragma unroll
      for (int k = 0; k < 3 * kVPT; ++k) uv[k] = 0.0f;
      if (nv == kVPT) {
        if (HIST) load4(F + lin0, fv);
        if (SAMPLE && a.u) {
          const float4* up = reinterpret_cast<const float4*>(a.u + 3ull * lin0);
          const float4 q0 = __ldg(up), q1 = __ldg(up + 1), q2 = __ldg(up + 2);
          uv[0] = q0.x; uv[1] = q0.y; uv[2] = q0.z; uv[3] = q0.w;
          uv[4] = q1.x; uv[5] = q1.y; uv[6] = q1.z; uv[7] = q1.w;
          uv[8] = q2.x; uv[9] = q2.y; uv[10] = q2.z; uv[11] = q2.w;
        }
        if (!SAMPLE) load4(a.Jin + lin0, jv);
      } else {
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          if ((unsigned)v < nv) {
            if (HIST) fv[v] = load1(F + lin0 + v);
            if (SAMPLE && a.u) {
              uv[3 * v + 0] = __ldg(a.u + 3ull * (lin0 + v) + 0);
              uv[3 * v + 1] = __ldg(a.u + 3ull * (lin0 + v) + 1);
              uv[3 * v + 2] = __ldg(a.u + 3ull * (lin0 + v) + 2);
            }
            if (!SAMPLE) jv[v] = __ldg(a.Jin + lin0 + v);
          }
        }
      }
      int ix, iy, iz;
      lin_to_xyz(g, lin0, ix, iy, iz);
      long long P[3];
      if (SAMPLE) anchor(g, ix, iy, iz, P);
#pragma unroll
      for (int v = 0; v < kVPT; ++v) {
        if (v > 0) {
          if (++ix == g.fW) {
            ix = 0;
            if (++iy == g.fH) {
              iy = 0;
              ++iz;
            }
            if (SAMPLE) anchor(g, ix, iy, iz, P);
          } else if (SAMPLE) {
            P[0] += g.Gq[0];
            P[1] += g.Gq[3];
            P[2] += g.Gq[6];
          }
        }
        if ((unsigned)v < nv) {
          if (SAMPLE) {
            int b[3];
            float r[3], d0, d1, d2;
            cell_of(g, P, uv[3 * v], uv[3 * v + 1], uv[3 * v + 2], b, r);
            jv[v] = trilinear<MT, false>(M, g, b, r, d0, d1, d2);
          }
          if (HIST) hist_add<BMAX>(hist_sm, a.bf, a.bj, fv[v], jv[v]);
        }
      }
      if (WRITEJ) {
        if (nv == kVPT) {
          *reinterpret_cast<float4*>(a.Jout + lin0) = make_float4(jv[0], jv[1], jv[2], jv[3]);
        } else {
#pragma unroll
          for (int v = 0; v < kVPT; ++v)
            if ((unsigned)v < nv) a.Jout[lin0 + v] = jv[v];
        }
      }
    }
    if (HIST && ++pending == kFlushEvery) {
      hist_flush<BMAX>(hist_sm, a.ghist, a.B);
      pending = 0;
    }
  }
  if (HIST) hist_flush<BMAX>(hist_sm, a.ghist, a.B);
}

// ------------------------------------------------------------ MI finalize
// One CTA: P = H / (N 2^kHistFrac); marginals as row / column sums of the
// joint (equal to the separately defined marginals by partition of unity);
// MI = sum_{P>0} P (ln P - ln P_F - ln P_J); packed table of the scaled T.
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
    P[i] = t;
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
  const double sc = a.tscale;
  for (int i = tid; i < nb; i += blockDim.x) {
    const int ra = i / B, rb = i - ra * B;
    auto T = [&](int bb) -> float { return bb < B ? (float)(P[ra * B + bb] * sc) : 0.0f; };
    if (BMAX == 32) {
      reinterpret_cast<float4*>(a.T)[ra * BMAX + rb] = make_float4(T(rb), T(rb + 1), T(rb + 2), T(rb + 3));
    } else {
      reinterpret_cast<float2*>(a.T)[ra * BMAX + rb] = make_float2(T(rb), T(rb + 1));
    }
  }
}

// ------------------------------------------------------------------ sweep 2
// Per voxel g = dL/dJ (MI table or a given buffer), then either dJ (MI on a
// materialised J) or the sampler backward: du = K^T (g dJ/dq) and the affine
// partial sums, reduced per CTA in fp64.
template <typename FT, typename MT, int BMAX, int MODE>
__global__ void __launch_bounds__(kThreads) k_sweep2(const Sweep2Args a) {
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
  float acc[12];
  double dacc[12];
#pragma unroll
  for (int k = 0; k < 12; ++k) {
    acc[k] = 0.0f;
    dacc[k] = 0.0;
  }
  int pending = 0;
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x) {
    const unsigned lin0 = (it * kThreads + threadIdx.x) * kVPT;
    if (lin0 < g.N) {
      const unsigned nv = min(g.N - lin0, (unsigned)kVPT);
      float fv[kVPT] = {0.f, 0.f, 0.f, 0.f}, jv[kVPT] = {0.f, 0.f, 0.f, 0.f};
      float gb[kVPT] = {0.f, 0.f, 0.f, 0.f}, uv[3 * kVPT], out[3 * kVPT];
#pragma unroll
      for (int k = 0; k < 3 * kVPT; ++k) {
        uv[k] = 0.0f;
        out[k] = 0.0f;
      }
      if (nv == kVPT) {
        if (MI) load4(F + lin0, fv);
        if (SAMPLE && a.u) {
          const float4* up = reinterpret_cast<const float4*>(a.u + 3ull * lin0);
          const float4 q0 = __ldg(up), q1 = __ldg(up + 1), q2 = __ldg(up + 2);
          uv[0] = q0.x; uv[1] = q0.y; uv[2] = q0.z; uv[3] = q0.w;
          uv[4] = q1.x; uv[5] = q1.y; uv[6] = q1.z; uv[7] = q1.w;
          uv[8] = q2.x; uv[9] = q2.y; uv[10] = q2.z; uv[11] = q2.w;
        }
        if (!SAMPLE) load4(a.Jin + lin0, jv);
        if (!MI) load4(a.gbuf + lin0, gb);
      } else {
#pragma unroll
        for (int v = 0; v < kVPT; ++v) {
          if ((unsigned)v < nv) {
            if (MI) fv[v] = load1(F + lin0 + v);
            if (SAMPLE && a.u) {
              uv[3 * v + 0] = __ldg(a.u + 3ull * (lin0 + v) + 0);
              uv[3 * v + 1] = __ldg(a.u + 3ull * (lin0 + v) + 1);
              uv[3 * v + 2] = __ldg(a.u + 3ull * (lin0 + v) + 2);
            }
            if (!SAMPLE) jv[v] = __ldg(a.Jin + lin0 + v);
            if (!MI) gb[v] = __ldg(a.gbuf + lin0 + v);
          }
        }
      }
      int ix, iy, iz;
      lin_to_xyz(g, lin0, ix, iy, iz);
      long long P[3];
      if (SAMPLE) anchor(g, ix, iy, iz, P);
#pragma unroll
      for (int v = 0; v < kVPT; ++v) {
        if (v > 0) {
          if (++ix == g.fW) {
            ix = 0;
            if (++iy == g.fH) {
              iy = 0;
              ++iz;
            }
            if (SAMPLE) anchor(g, ix, iy, iz, P);
          } else if (SAMPLE) {
            P[0] += g.Gq[0];
            P[1] += g.Gq[3];
            P[2] += g.Gq[6];
          }
        }
        if ((unsigned)v < nv) {
          float j = jv[v], gq0 = 0.f, gq1 = 0.f, gq2 = 0.f;
          if (SAMPLE) {
            int b[3];
            float r[3];
            cell_of(g, P, uv[3 * v], uv[3 * v + 1], uv[3 * v + 2], b, r);
            j = trilinear<MT, true>(M, g, b, r, gq0, gq1, gq2);
          }
          const float gv = MI ? mi_grad<BMAX>(tsm, a.bf, a.bj, fv[v], j) : gb[v];
          if (BWD) {
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
          } else {
            out[v] = gv;
          }
        }
      }
      if (BWD) {
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
        dacc[k] += (double)warp_sum(acc[k]);
        acc[k] = 0.0f;
      }
      pending = 0;
    }
  }
  if (BWD) {
#pragma unroll
    for (int k = 0; k < 12; ++k) dacc[k] += (double)warp_sum(acc[k]);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
#pragma unroll
      for (int k = 0; k < 12; ++k) wsum[w][k] = dacc[k];
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

template <typename FT, typename MT, int BMAX, int MODE>
static size_t sweep1_smem() {
  return MODE == S1_WRITEJ ? 0 : (size_t)BMAX * (BMAX + 8) * sizeof(unsigned);
}

template <typename FT, typename MT, int BMAX, int MODE>
static cudaError_t run_sweep1(const Sweep1Args& a, int grid, cudaStream_t s, int* occ) {
  auto k = k_sweep1<FT, MT, BMAX, MODE>;
  const size_t smem = sweep1_smem<FT, MT, BMAX, MODE>();
  if (occ) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kThreads, smem);
    return e;
  }
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

}  // namespace ffdp
