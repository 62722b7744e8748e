// k_lncc.cu -- fused LNCC forward + backward on a materialised warped image J,
// optionally fused with the MI partial gradient and the sampler backward.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration", Key designs item 2: all LNCC intermediates (the window sums
// of I, J, I^2, J^2, IJ) stay on chip.  Definition used (zero padding, window
// w = 2R+1, n = w^3):
//   cross = S_FJ - S_F S_J / n,  vF = S_FF - S_F^2 / n,  vJ = S_JJ - S_J^2 / n,
//   cc = cross^2 / (vF vJ + eps),  LNCC = mean(cc),
//   with D = vF vJ + eps, A1 = 2 cross / D, A2 = cross^2 vF / D^2 and
//   s = -w_lncc / N:  g_FJ = s A1,  g_JJ = -s A2,  g_J = s (2 A2 S_J - A1 S_F) / n,
//   dJ_m = sum_{k in window(m)} g_J(k) + 2 J_m g_JJ(k) + F_m g_FJ(k).
//
// Work layout: a CTA owns a 32 x TY column of output voxels and streams a
// z-range of planes through shared memory.  Per incoming plane: the (J, F)
// plane with a 2R halo enters a ring of w planes; the 5 products are summed
// over the ring (z), then along x and y, giving the window sums one plane
// behind; the three g-terms enter a second ring, are summed the same way and
// give dJ 2R planes behind the incoming plane.  CTAs are persistent over
// tiles, so the per-CTA partial records stay O(#SMs).
#include "ffdp_internal.h"

namespace ffdp {

constexpr int kTX = kLnccTX;

struct LnccLayout {
  int W_, TY, E2W, E2H, E1W, E1H, E2, E1;
  int off_jf, off_zb, off_xb, off_gr, off_T, total;
};

__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

__host__ __device__ inline LnccLayout lncc_layout(int R, int bmax) {
  LnccLayout L;
  L.W_ = 2 * R + 1;
  L.TY = R <= 2 ? 16 : 8;
  L.E2W = kTX + 4 * R;
  L.E2H = L.TY + 4 * R;
  L.E1W = kTX + 2 * R;
  L.E1H = L.TY + 2 * R;
  L.E2 = L.E2W * L.E2H;
  L.E1 = L.E1W * L.E1H;
  L.off_jf = 0;
  L.off_zb = L.off_jf + L.W_ * L.E2 * 2;
  L.off_xb = L.off_zb + imax(5 * L.E2, 3 * L.E1);
  L.off_gr = L.off_xb + imax(5 * L.E2H * L.E1W, 3 * L.E1H * kTX);
  L.off_T = ((L.off_gr + L.W_ * 3 * L.E1) + 3) & ~3;
  const int tf = bmax * bmax * 2;
  L.total = L.off_T + tf;
  return L;
}

size_t lncc_smem_bytes(int R, int bmax_or0) { return (size_t)lncc_layout(R, bmax_or0).total * sizeof(float); }

// MI partial gradient from T rows packed as float2 pairs (any bin count).
template <int BMAX>
__device__ __forceinline__ float mi_grad_ln(const float* tsm, const BinMap& bf, const BinMap& bj, float f,
                                            float j) {
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float wf[4], d[4];
  bspline4(tf, 1.0f, wf);
  bspline4_deriv(tj, d);
  float s = 0.0f;
  const float2* t2 = reinterpret_cast<const float2*>(tsm) + (af - 1) * BMAX + (aj - 1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = t2[i * BMAX], q = t2[i * BMAX + 2];
    s = fmaf(wf[i], fmaf(p.x, d[0], fmaf(p.y, d[1], fmaf(q.x, d[2], q.y * d[3]))), s);
  }
  return (j >= bj.lo && j <= bj.hi) ? s : 0.0f;
}

template <typename FT, typename MT, int MODE, int BMAX>
__global__ void __launch_bounds__(kThreads) k_lncc(const LnccArgs a) {
  constexpr bool MI = BMAX != 0;
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ double wsum[kThreads / 32][13];
  const int R = a.R;
  const LnccLayout L = lncc_layout(R, BMAX);
  const Geom& g = a.g;
  const int W_ = L.W_, TY = L.TY, E2W = L.E2W, E2H = L.E2H, E1W = L.E1W, E1H = L.E1H;
  const int E2 = L.E2, E1 = L.E1;
  float2* jf = reinterpret_cast<float2*>(sm + L.off_jf);
  float* zb = sm + L.off_zb;
  float* xb = sm + L.off_xb;
  float* gr = sm + L.off_gr;
  float* tsm = sm + L.off_T;
  const int tid = threadIdx.x;
  if (MI) {
    const int n4 = BMAX * BMAX * 2 / 4;
    const float4* src = reinterpret_cast<const float4*>(a.T);
    for (int i = tid; i < n4; i += kThreads) reinterpret_cast<float4*>(tsm)[i] = __ldg(src + i);
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  const float inv_n = a.inv_n, eps = a.eps, gs = a.gscale;
  float cc_acc = 0.0f;
  float acc[12];
#pragma unroll
  for (int k = 0; k < 12; ++k) acc[k] = 0.0f;
  double dacc[13];
#pragma unroll
  for (int k = 0; k < 13; ++k) dacc[k] = 0.0;

  const int chunksZ = (g.fD + a.tz - 1) / a.tz;
  const int ntiles = a.tilesX * a.tilesY * chunksZ;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    int t = tile;
    const int tx = t % a.tilesX;
    t /= a.tilesX;
    const int ty = t % a.tilesY;
    const int tzc = t / a.tilesY;
    const int x0 = tx * kTX, y0 = ty * TY, z0 = tzc * a.tz;
    const int z1 = min(z0 + a.tz, g.fD);
    const int nsteps = (z1 - z0) + 4 * R;
    for (int s = 0; s < nsteps; ++s) {
      const int zi = z0 - 2 * R + s;
      // [A] incoming (J, F) plane with a 2R halo; zero outside the grid.
      {
        float2* slot = jf + (s % W_) * E2;
        const bool zin = zi >= 0 && zi < g.fD;
        for (int e = tid; e < E2; e += kThreads) {
          const int ey = e / E2W, ex = e - ey * E2W;
          const int x = x0 - 2 * R + ex, y = y0 - 2 * R + ey;
          float2 v = make_float2(0.0f, 0.0f);
          if (zin && (unsigned)x < (unsigned)g.fW && (unsigned)y < (unsigned)g.fH) {
            const size_t lin = ((size_t)zi * g.fH + y) * g.fW + x;
            v.x = __ldg(a.J + lin);
            v.y = load1(F + lin);
          }
          slot[e] = v;
        }
      }
      __syncthreads();
      if (s >= 2 * R) {
        // [B] z sums of F, J, F^2, J^2, FJ over the ring (planes zi-2R .. zi).
        for (int e = tid; e < E2; e += kThreads) {
          float sF = 0.f, sJ = 0.f, sFF = 0.f, sJJ = 0.f, sFJ = 0.f;
          for (int k = 0; k < W_; ++k) {
            const float2 v = jf[k * E2 + e];
            sJ += v.x;
            sF += v.y;
            sJJ = fmaf(v.x, v.x, sJJ);
            sFF = fmaf(v.y, v.y, sFF);
            sFJ = fmaf(v.x, v.y, sFJ);
          }
          zb[0 * E2 + e] = sF;
          zb[1 * E2 + e] = sJ;
          zb[2 * E2 + e] = sFF;
          zb[3 * E2 + e] = sJJ;
          zb[4 * E2 + e] = sFJ;
        }
        __syncthreads();
        // [C] x sums: E2H rows, E1W outputs per row.
        for (int e = tid; e < E2H * E1W; e += kThreads) {
          const int row = e / E1W, x1 = e - row * E1W;
#pragma unroll
          for (int q = 0; q < 5; ++q) {
            const float* src = zb + q * E2 + row * E2W + x1;
            float sacc = 0.0f;
            for (int k = 0; k <= 2 * R; ++k) sacc += src[k];
            xb[q * E2H * E1W + e] = sacc;
          }
        }
        __syncthreads();
        // [D] y sums give the window sums at plane zc on the R-halo region;
        // cc and the three g-terms (zero outside the grid).
        {
          const int zc = zi - R;
          float* gslot = gr + (s % W_) * 3 * E1;
          const bool zin = zc >= 0 && zc < g.fD;
          const bool zown = zc >= z0 && zc < z1;
          for (int e = tid; e < E1; e += kThreads) {
            const int y1 = e / E1W, x1 = e - y1 * E1W;
            float S[5];
#pragma unroll
            for (int q = 0; q < 5; ++q) {
              const float* src = xb + q * E2H * E1W + y1 * E1W + x1;
              float sacc = 0.0f;
              for (int k = 0; k <= 2 * R; ++k) sacc += src[k * E1W];
              S[q] = sacc;
            }
            const int x = x0 - R + x1, y = y0 - R + y1;
            float gJ = 0.f, gJJ = 0.f, gFJ = 0.f;
            if (zin && (unsigned)x < (unsigned)g.fW && (unsigned)y < (unsigned)g.fH) {
              const float cross = fmaf(-S[0] * S[1], inv_n, S[4]);
              const float vF = fmaf(-S[0] * S[0], inv_n, S[2]);
              const float vJ = fmaf(-S[1] * S[1], inv_n, S[3]);
              const float D = fmaf(vF, vJ, eps);
              const float rD = 1.0f / D;
              const float A1 = 2.0f * cross * rD;
              const float cc = cross * cross * rD;
              const float A2 = cc * vF * rD;
              gFJ = gs * A1;
              gJJ = -gs * A2;
              gJ = gs * (2.0f * A2 * S[1] - A1 * S[0]) * inv_n;
              if (zown && x1 >= R && x1 < R + kTX && y1 >= R && y1 < R + TY) cc_acc += cc;
            }
            gslot[e] = gJ;
            gslot[E1 + e] = gJJ;
            gslot[2 * E1 + e] = gFJ;
          }
        }
        __syncthreads();
      }
      if (s >= 4 * R) {
        // [E] z sums of the g-terms over their ring.
        float* gz = zb;
        for (int e = tid; e < E1; e += kThreads) {
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            float sacc = 0.0f;
            for (int k = 0; k < W_; ++k) sacc += gr[k * 3 * E1 + c * E1 + e];
            gz[c * E1 + e] = sacc;
          }
        }
        __syncthreads();
        // [F] x sums onto the 32 output columns.
        float* gx = xb;
        for (int e = tid; e < E1H * kTX; e += kThreads) {
          const int row = e / kTX, x = e - row * kTX;
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const float* src = gz + c * E1 + row * E1W + x;
            float sacc = 0.0f;
            for (int k = 0; k <= 2 * R; ++k) sacc += src[k];
            gx[c * E1H * kTX + e] = sacc;
          }
        }
        __syncthreads();
        // [G] y sums at the outputs of plane zo, then the epilogue.
        {
          const int zo = zi - 2 * R;
          const float2* jfo = jf + ((s - 2 * R) % W_) * E2;
          for (int e = tid; e < kTX * TY; e += kThreads) {
            const int yy = e / kTX, xx = e - yy * kTX;
            const int X = x0 + xx, Y = y0 + yy;
            if (X < g.fW && Y < g.fH) {
              float bg[3];
#pragma unroll
              for (int c = 0; c < 3; ++c) {
                const float* src = gx + c * E1H * kTX + yy * kTX + xx;
                float sacc = 0.0f;
                for (int k = 0; k <= 2 * R; ++k) sacc += src[k * kTX];
                bg[c] = sacc;
              }
              const float2 v = jfo[(yy + 2 * R) * E2W + (xx + 2 * R)];
              float gv = fmaf(v.y, bg[2], fmaf(2.0f * v.x, bg[1], bg[0]));
              if (MI) gv += mi_grad_ln<(MI ? BMAX : 32)>(tsm, a.bf, a.bj, v.y, v.x);
              const size_t lin = ((size_t)zo * g.fH + Y) * g.fW + X;
              if (MODE == LN_DJ) {
                if (a.dJ) a.dJ[lin] = gv;
              } else {
                long long P[3];
                anchor(g, X, Y, zo, P);
                float u0 = 0.f, u1 = 0.f, u2 = 0.f;
                if (a.u) {
                  u0 = __ldg(a.u + 3 * lin + 0);
                  u1 = __ldg(a.u + 3 * lin + 1);
                  u2 = __ldg(a.u + 3 * lin + 2);
                }
                int b[3];
                float r[3], gq0, gq1, gq2;
                cell_of(g, P, u0, u1, u2, b, r);
                trilinear<MT, true>(M, g, b, r, gq0, gq1, gq2);
                const float e0 = gv * gq0, e1 = gv * gq1, e2 = gv * gq2;
                if (a.du) {
                  if (g.k_diag) {
                    a.du[3 * lin + 0] = g.K[0] * e0;
                    a.du[3 * lin + 1] = g.K[4] * e1;
                    a.du[3 * lin + 2] = g.K[8] * e2;
                  } else {
                    a.du[3 * lin + 0] = fmaf(g.K[0], e0, fmaf(g.K[3], e1, g.K[6] * e2));
                    a.du[3 * lin + 1] = fmaf(g.K[1], e0, fmaf(g.K[4], e1, g.K[7] * e2));
                    a.du[3 * lin + 2] = fmaf(g.K[2], e0, fmaf(g.K[5], e1, g.K[8] * e2));
                  }
                }
                const float cx = (float)X - g.ctr[0], cy = (float)Y - g.ctr[1], cz = (float)zo - g.ctr[2];
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
          }
        }
        __syncthreads();
      }
      // fold the fp32 partials into fp64 every 8 planes (uniform across the CTA)
      if ((s & 7) == 7) {
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          dacc[k] += (double)warp_sum(acc[k]);
          acc[k] = 0.0f;
        }
        dacc[12] += (double)warp_sum(cc_acc);
        cc_acc = 0.0f;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 12; ++k) dacc[k] += (double)warp_sum(acc[k]);
  dacc[12] += (double)warp_sum(cc_acc);
  const int w = tid >> 5;
  if ((tid & 31) == 0)
#pragma unroll
    for (int k = 0; k < 13; ++k) wsum[w][k] = dacc[k];
  __syncthreads();
  if (tid < kPartialStride) {
    double s = 0.0;
    if (tid < 13)
      for (int k = 0; k < kThreads / 32; ++k) s += wsum[k][tid];
    a.partials[(size_t)blockIdx.x * kPartialStride + tid] = s;
  }
}

// occ != nullptr: report resident CTAs per SM instead of launching.
template <typename FT, typename MT, int MODE, int BMAX>
static cudaError_t run_lncc(const LnccArgs& a, int grid, cudaStream_t s, int R, int* occ) {
  auto k = k_lncc<FT, MT, MODE, BMAX>;
  const size_t smem = lncc_smem_bytes(R, BMAX);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kThreads, smem);
  note_launch_begin("k_lncc", s);
  k<<<grid, kThreads, smem, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

static cudaError_t dispatch_lncc(int mode, int ft, int mt, int bmax, const LnccArgs& a, int grid,
                                 cudaStream_t s, int R, int* occ) {
  cudaError_t e = cudaErrorInvalidValue;
  FFDP_DT_SWITCH(ft, FT, FFDP_DT_SWITCH(mt, MT, {
    if (mode == LN_DJ) {
      e = run_lncc<FT, float, LN_DJ, 0>(a, grid, s, R, occ);
    } else if (bmax == 0) {
      e = run_lncc<FT, MT, LN_BWD, 0>(a, grid, s, R, occ);
    } else if (bmax == 32) {
      e = run_lncc<FT, MT, LN_BWD, 32>(a, grid, s, R, occ);
    } else {
      e = run_lncc<FT, MT, LN_BWD, 64>(a, grid, s, R, occ);
    }
  }));
  return e;
}

cudaError_t launch_lncc(int mode, int ft, int mt, int bmax, const LnccArgs& a, int grid, cudaStream_t s) {
  return dispatch_lncc(mode, ft, mt, bmax, a, grid, s, a.R, nullptr);
}

int lncc_ctas_per_sm(int mode, int ft, int mt, int bmax, int R) {
  int occ = 0;
  LnccArgs dummy{};
  if (dispatch_lncc(mode, ft, mt, bmax, dummy, 0, 0, R, &occ) != cudaSuccess || occ < 1) occ = 1;
  return occ > kMaxCtasPerSm ? kMaxCtasPerSm : occ;
}

}  // namespace ffdp
