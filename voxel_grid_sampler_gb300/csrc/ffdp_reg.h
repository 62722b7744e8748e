// ffdp_reg.h -- argument record and launcher of the regularised update
// (Sobolev regulariser + Adam step of u), shared by the host ABI and k_reg.cu.
#pragma once

#include "ffdp_internal.h"

namespace ffdp {

// Sobolev regulariser of u ([N][3], channel-last) and, in the step mode, the
// Adam update u_out = u - lr m1^ / (sqrt(m2^) + eps) with G = g + dR/du.
struct RegArgs {
  const float* u;
  float* dR;          // regulariser mode: [N][3] gradient or NULL
  const float* g;     // step mode: [N][3] objective gradient (du)
  float* u_out;       // step mode: [N][3], must not overlap u
  float* m1;          // step mode: [N][3], updated in place
  float* m2;
  double* partials;   // [gridDim.x][kPartialStride]: slot kPSE = lambda sum of squared forward differences
  Geom g3;            // fixed-grid extents and fast-division constants
  float coef;         // 2 lambda / N
  float lambda;
  float lr, b1, b2, eps;
  float ic1, ic2;     // 1 / (1 - b1^t), 1 / (1 - b2^t)
};

constexpr int kRegThreads = 256;
cudaError_t launch_reg(int step, const RegArgs& a, int grid, cudaStream_t s);
int reg_ctas_per_sm(int step);

}  // namespace ffdp
