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
// Work layout: a persistent grid of kRegThreads-thread CTAs strides over
// warp-uniform groups of 32 consecutive voxels.  A lane's x neighbours are
// its neighbouring lanes' own u (shuffles; the group's two end lanes load
// theirs), the y and z neighbours come from L1 / L2 (the rows and planes
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

cudaError_t launch_reg(int step, const RegArgs& a, int grid, cudaStream_t s) {
  note_launch_begin(step ? "k_reg_adam" : "k_reg", s);
  if (step)
    k_reg<1><<<grid, kRegThreads, 0, s>>>(a);
  else
    k_reg<0><<<grid, kRegThreads, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

int reg_ctas_per_sm(int step) {
  static int cache[2] = {0, 0};
  int& c = cache[step ? 1 : 0];
  if (c == 0) {
    int occ = 0;
    const cudaError_t e = step ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_reg<1>, kRegThreads, 0)
                               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_reg<0>, kRegThreads, 0);
    if (e != cudaSuccess || occ < 1) occ = 1;
    c = occ > kMaxCtasPerSm ? kMaxCtasPerSm : occ;
  }
  return c;
}

}  // namespace ffdp
