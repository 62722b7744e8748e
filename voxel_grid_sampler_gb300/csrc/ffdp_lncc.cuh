// ffdp_lncc.cuh -- device helpers shared by the LNCC window kernels (the
// tiled kernels of k_lncc.cu and the wide-window passes of k_lncc_wide.cu).
#pragma once

#include "ffdp_internal.h"

namespace ffdp {

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// MI partial gradient from the polynomial cells of the MI table (global,
// read through L1): per cell (floor cF, floor cJ) the 12 coefficients of the
// bicubic-in-tF, biquadratic-in-tJ polynomial sum_{a,b} T beta beta'.
template <int BMAX>
__device__ __forceinline__ float mi_grad_ln(const float* __restrict__ T, const BinMap& bf, const BinMap& bj,
                                            float f, float j) {
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  const float4* c = reinterpret_cast<const float4*>(T) + 3 * (af * BMAX + aj);
  const float4 c0 = __ldg(c), c1 = __ldg(c + 1), c2 = __ldg(c + 2);
  // coefficients C[p][r] of tF^p tJ^r: c0 = (C00, C01, C02, C10), c1 = (C11, C12, C20, C21),
  // c2 = (C22, C30, C31, C32)
  const float p0 = fmaf(fmaf(c0.z, tj, c0.y), tj, c0.x);
  const float p1 = fmaf(fmaf(c1.y, tj, c1.x), tj, c0.w);
  const float p2 = fmaf(fmaf(c2.x, tj, c1.w), tj, c1.z);
  const float p3 = fmaf(fmaf(c2.w, tj, c2.z), tj, c2.y);
  const float s = fmaf(fmaf(fmaf(p3, tf, p2), tf, p1), tf, p0);
  return (j >= bj.lo && j <= bj.hi) ? s : 0.0f;
}

}  // namespace ffdp
