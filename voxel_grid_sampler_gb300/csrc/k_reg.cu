// k_reg.cu -- the regulariser term R(phi) of the objective and the optimiser
// step of the displacement field, fused into one pass over u.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration".  "Background": L(phi) = C(F, M o phi) + R(phi) with R a
// Sobolev norm; the overview updates the warp by gradient descent with
// optimiser state [m1], [m2] held per voxel beside u (which Grid Parallel
// shards with u).  Definitions used (the page gives none):
//   R(u) = (lambda / N) sum_c sum_a sum_{i: i + e_a inside} (u_c(i + e_a) - u_c(i))^2,
//   dR/du_c(i) = (2 lambda / N) sum_{j neighbour of i, inside} (u_c(i) - u_c(j)),
// and Adam with bias correction on G = du + dR/du:
//   m1 = b1 m1 + (1 - b1) G,  m2 = b2 m2 + (1 - b2) G^2,
//   u_out = u - lr (m1 / (1 - b1^t)) / (sqrt(m2 / (1 - b2^t)) + eps).
//
// Work layout: a persistent grid of kRegThreads-thread CTAs.  Two forms with
// the same arithmetic: where W and N are multiples of 4, k_reg_v moves the
// flat [N][3] arrays as one 16-byte vector per lane (below); otherwise k_reg
// strides over warp-uniform groups of 32 consecutive voxels.  In both, x
// neighbours come from the neighbouring lanes (shuffles; the end lanes
// load theirs) and the y and z neighbours from L1 / L2 (the rows and planes
// around the sweeping front stay resident), so u is read from HBM once; g,
// m1, m2 stream once and u_out, m1, m2 are written once: 84 bytes per voxel
// in the step mode.  The energy is summed per thread in fp32, folded into
// per-warp fp64 sums every kRegFold groups, then per CTA.
#include "ffdp_reg.h"

namespace ffdp {

constexpr int kRegFold = 32;

__device__ __forceinline__ void ld3(const float* __restrict__ p, unsigned long long i, float v[3]) {
  v[0] = __ldg(p + 3 * i + 0);
  v[1] = __ldg(p + 3 * i + 1);
  v[2] = __ldg(p + 3 * i + 2);
}

template <int STEP>
__global__ void __launch_bounds__(kRegThreads, 4) k_reg(const RegArgs a) {
  __shared__ double wsum[kRegThreads / 32];
  const Geom& g = a.g3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wsum[warp] = 0.0;
  float acc = 0.0f;
  int pend = 0;
  const unsigned long long HW = (unsigned long long)g.fW * g.fH;
  const unsigned long long stride = (unsigned long long)gridDim.x * kRegThreads;
  for (unsigned long long l0 = (unsigned long long)blockIdx.x * kRegThreads + 32 * warp; l0 < g.N; l0 += stride) {
    const bool act = l0 + lane < g.N;
    const unsigned lin = act ? (unsigned)(l0 + lane) : (unsigned)(g.N - 1);
    int x, y, z;
    lin_to_xyz(g, lin, x, y, z);
    float u0[3];
    ld3(a.u, lin, u0);
    // x neighbours: the neighbouring lanes hold voxels lin -/+ 1
    float ul[3], ur[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      ul[c] = __shfl_up_sync(0xffffffffu, u0[c], 1);
      ur[c] = __shfl_down_sync(0xffffffffu, u0[c], 1);
    }
    const bool hasl = x > 0, hasr = x + 1 < g.fW;
    if (act) {
      if (lane == 0 && hasl) ld3(a.u, lin - 1ull, ul);
      if ((lane == 31 || l0 + lane + 1 >= g.N) && hasr) ld3(a.u, lin + 1ull, ur);
      float d[3] = {0.0f, 0.0f, 0.0f}, s = 0.0f;  // d: sum over neighbours of (u_j - u_i)
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        if (hasl) d[c] += ul[c] - u0[c];
        if (hasr) {
          const float e = ur[c] - u0[c];
          d[c] += e;
          s = fmaf(e, e, s);
        }
      }
      float v[3];
      if (y > 0) {
        ld3(a.u, lin - (unsigned long long)g.fW, v);
#pragma unroll
        for (int c = 0; c < 3; ++c) d[c] += v[c] - u0[c];
      }
      if (y + 1 < g.fH) {
        ld3(a.u, lin + (unsigned long long)g.fW, v);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const float e = v[c] - u0[c];
          d[c] += e;
          s = fmaf(e, e, s);
        }
      }
      if (z > 0) {
        ld3(a.u, lin - HW, v);
#pragma unroll
        for (int c = 0; c < 3; ++c) d[c] += v[c] - u0[c];
      }
      if (z + 1 < g.fD) {
        ld3(a.u, lin + HW, v);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const float e = v[c] - u0[c];
          d[c] += e;
          s = fmaf(e, e, s);
        }
      }
      acc += s;
      float gr[3];
#pragma unroll
      for (int c = 0; c < 3; ++c) gr[c] = -a.coef * d[c];  // dR/du
      const unsigned long long o = 3ull * lin;
      if constexpr (STEP == 0) {
        if (a.dR) {
          a.dR[o + 0] = gr[0];
          a.dR[o + 1] = gr[1];
          a.dR[o + 2] = gr[2];
        }
      } else {
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const float G = __ldg(a.g + o + c) + gr[c];
          const float m1 = fmaf(a.b1, a.m1[o + c], (1.0f - a.b1) * G);
          const float m2 = fmaf(a.b2, a.m2[o + c], (1.0f - a.b2) * G * G);
          a.m1[o + c] = m1;
          a.m2[o + c] = m2;
          a.u_out[o + c] = u0[c] - a.lr * (m1 * a.ic1) / (sqrtf(m2 * a.ic2) + a.eps);
        }
      }
    }
    if (++pend == kRegFold) {
      const float t = warp_sum(acc);
      if (lane == 0) wsum[warp] += (double)t;
      acc = 0.0f;
      pend = 0;
    }
  }
  {
    const float t = warp_sum(acc);
    if (lane == 0) wsum[warp] += (double)t;
  }
  __syncthreads();
  if (threadIdx.x < kPartialStride) {
    double s = 0.0;
    if (threadIdx.x == kPSE)
      for (int w = 0; w < kRegThreads / 32; ++w) s += wsum[w];
    a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = s * (double)a.lambda;
  }
}

// Vector form for grids with W and N multiples of 4 (then 3W and 3N are too):
// u, g, m1, m2, u_out and dR are read and written as the flat float arrays
// they are ([N][3] = 3N floats), one aligned 16-byte vector per lane, so every
// warp access is 512 contiguous bytes.  Element f = 4 q + j of vector q is
// channel f mod 3 of voxel f / 3; its x neighbours are elements f -/+ 3 (the
// same vector or the neighbouring lane's, by shuffles; the warp's end lanes
// load the next vector), its y and z neighbours the same lane of the vectors
// 3W/4 and 3HW/4 away (aligned because W is a multiple of 4).  A vector holds
// elements of at most two voxels (v0 and v0 + 1).
template <int STEP>
__global__ void __launch_bounds__(kRegThreads, 4) k_reg_v(const RegArgs a) {
  __shared__ double wsum[kRegThreads / 32];
  const Geom& g = a.g3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wsum[warp] = 0.0;
  float acc = 0.0f;
  int pend = 0;
  const unsigned long long NQ = 3ull * g.N / 4;  // vectors
  const unsigned long long QY = 3ull * g.fW / 4, QZ = QY * g.fH;
  const float4* __restrict__ u4 = reinterpret_cast<const float4*>(a.u);
  const unsigned long long stride = (unsigned long long)gridDim.x * kRegThreads;
  for (unsigned long long q0 = (unsigned long long)blockIdx.x * kRegThreads + 32 * warp; q0 < NQ; q0 += stride) {
    const unsigned long long q = q0 + lane;
    const bool act = q < NQ;
    float4 U = make_float4(0.f, 0.f, 0.f, 0.f);
    if (act) U = __ldg(u4 + q);
    // x neighbours across lanes: elements 1..3 of the vector below, 0..2 of the one above
    float dn[3], up[3];
    dn[0] = __shfl_up_sync(0xffffffffu, U.y, 1);
    dn[1] = __shfl_up_sync(0xffffffffu, U.z, 1);
    dn[2] = __shfl_up_sync(0xffffffffu, U.w, 1);
    up[0] = __shfl_down_sync(0xffffffffu, U.x, 1);
    up[1] = __shfl_down_sync(0xffffffffu, U.y, 1);
    up[2] = __shfl_down_sync(0xffffffffu, U.z, 1);
    if (act) {
      if (lane == 0 && q > 0) {
        const float4 B = __ldg(u4 + q - 1);
        dn[0] = B.y;
        dn[1] = B.z;
        dn[2] = B.w;
      }
      if ((lane == 31 || q + 1 >= NQ) && q + 1 < NQ) {
        const float4 B = __ldg(u4 + q + 1);
        up[0] = B.x;
        up[1] = B.y;
        up[2] = B.z;
      }
      // voxel of the vector's first element and its coordinates; the next voxel's
      const unsigned long long f0 = 4ull * q;
      const unsigned v0 = (unsigned)(__umul64hi(f0, 0xAAAAAAAAAAAAAAABull) >> 1);  // f0 / 3
      const int c0 = (int)(f0 - 3ull * v0);
      int x0, y0, z0, x1, y1, z1;
      lin_to_xyz(g, v0, x0, y0, z0);
      if (x0 + 1 < g.fW) {
        x1 = x0 + 1;
        y1 = y0;
        z1 = z0;
      } else {
        lin_to_xyz(g, v0 + 1 < g.N ? v0 + 1 : v0, x1, y1, z1);
      }
      float4 Ym = make_float4(0.f, 0.f, 0.f, 0.f), Yp = Ym, Zm = Ym, Zp = Ym;
      if (q >= QY) Ym = __ldg(u4 + q - QY);
      if (q + QY < NQ) Yp = __ldg(u4 + q + QY);
      if (q >= QZ) Zm = __ldg(u4 + q - QZ);
      if (q + QZ < NQ) Zp = __ldg(u4 + q + QZ);
      const float uu[4] = {U.x, U.y, U.z, U.w};
      const float ym[4] = {Ym.x, Ym.y, Ym.z, Ym.w}, yp[4] = {Yp.x, Yp.y, Yp.z, Yp.w};
      const float zm[4] = {Zm.x, Zm.y, Zm.z, Zm.w}, zp[4] = {Zp.x, Zp.y, Zp.z, Zp.w};
      // elements f -/+ 3: xl[j], xr[j]
      const float xl[4] = {dn[0], dn[1], dn[2], uu[0]};
      const float xr[4] = {uu[3], up[0], up[1], up[2]};
      float gr[4], s = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool second = c0 + j >= 3;  // element of voxel v0 + 1
        const int x = second ? x1 : x0, y = second ? y1 : y0, z = second ? z1 : z0;
        float d = 0.0f;
        if (x > 0) d += xl[j] - uu[j];
        if (x + 1 < g.fW) {
          const float e = xr[j] - uu[j];
          d += e;
          s = fmaf(e, e, s);
        }
        if (y > 0) d += ym[j] - uu[j];
        if (y + 1 < g.fH) {
          const float e = yp[j] - uu[j];
          d += e;
          s = fmaf(e, e, s);
        }
        if (z > 0) d += zm[j] - uu[j];
        if (z + 1 < g.fD) {
          const float e = zp[j] - uu[j];
          d += e;
          s = fmaf(e, e, s);
        }
        gr[j] = -a.coef * d;
      }
      acc += s;
      if constexpr (STEP == 0) {
        if (a.dR) reinterpret_cast<float4*>(a.dR)[q] = make_float4(gr[0], gr[1], gr[2], gr[3]);
      } else {
        const float4 G4 = __ldg(reinterpret_cast<const float4*>(a.g) + q);
        const float4 A4 = reinterpret_cast<const float4*>(a.m1)[q];
        const float4 B4 = reinterpret_cast<const float4*>(a.m2)[q];
        const float gg[4] = {G4.x, G4.y, G4.z, G4.w}, m1o[4] = {A4.x, A4.y, A4.z, A4.w};
        const float m2o[4] = {B4.x, B4.y, B4.z, B4.w};
        float n1[4], n2[4], uo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float G = gg[j] + gr[j];
          n1[j] = fmaf(a.b1, m1o[j], (1.0f - a.b1) * G);
          n2[j] = fmaf(a.b2, m2o[j], (1.0f - a.b2) * G * G);
          uo[j] = uu[j] - a.lr * (n1[j] * a.ic1) / (sqrtf(n2[j] * a.ic2) + a.eps);
        }
        reinterpret_cast<float4*>(a.m1)[q] = make_float4(n1[0], n1[1], n1[2], n1[3]);
        reinterpret_cast<float4*>(a.m2)[q] = make_float4(n2[0], n2[1], n2[2], n2[3]);
        reinterpret_cast<float4*>(a.u_out)[q] = make_float4(uo[0], uo[1], uo[2], uo[3]);
      }
    }
    if (++pend == kRegFold) {
      const float t = warp_sum(acc);
      if (lane == 0) wsum[warp] += (double)t;
      acc = 0.0f;
      pend = 0;
    }
  }
  {
    const float t = warp_sum(acc);
    if (lane == 0) wsum[warp] += (double)t;
  }
  __syncthreads();
  if (threadIdx.x < kPartialStride) {
    double s = 0.0;
    if (threadIdx.x == kPSE)
      for (int w = 0; w < kRegThreads / 32; ++w) s += wsum[w];
    a.partials[(size_t)blockIdx.x * kPartialStride + threadIdx.x] = s * (double)a.lambda;
  }
}

// The vector form runs where the grid allows it (W and N multiples of 4).
static bool reg_vector_form(const RegArgs& a) { return (a.g3.fW & 3) == 0 && (a.g3.N & 3u) == 0; }

cudaError_t launch_reg(int step, const RegArgs& a, int grid, cudaStream_t s) {
  note_launch_begin(step ? "k_reg_adam" : "k_reg", s);
  const bool vec = reg_vector_form(a);
  if (step)
    vec ? k_reg_v<1><<<grid, kRegThreads, 0, s>>>(a) : k_reg<1><<<grid, kRegThreads, 0, s>>>(a);
  else
    vec ? k_reg_v<0><<<grid, kRegThreads, 0, s>>>(a) : k_reg<0><<<grid, kRegThreads, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

int reg_ctas_per_sm(int step) {
  static OccCache<2> cache;
  return cache.get(step ? 1 : 0, [&] {
    // both forms are bounded to 64 registers (four 256-thread CTAs per SM); take the smaller occupancy
    int o1 = 0, o2 = 0;
    const cudaError_t e1 = step ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, k_reg<1>, kRegThreads, 0)
                                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, k_reg<0>, kRegThreads, 0);
    const cudaError_t e2 = step ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, k_reg_v<1>, kRegThreads, 0)
                                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, k_reg_v<0>, kRegThreads, 0);
    return (e1 == cudaSuccess && e2 == cudaSuccess) ? (o1 < o2 ? o1 : o2) : 1;
  });
}

}  // namespace ffdp
