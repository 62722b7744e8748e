/*
 * ffdp_oracle.c -- plain, slow, double-precision CPU oracle for the FFDP
 * registration objective (composite implicit grid sampler, Mattes mutual
 * information with a cubic B-spline Parzen window, local normalised cross
 * correlation) and its gradient with respect to u, A and t.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library: every quantity is computed
 * here straight from its definition, voxel by voxel, in double precision,
 * with no blocking, fusion or algebraic shortcut.
 *
 * Source: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
 * Registration" (ICLR 2026), as summarised on the papernotes.org page of that
 * title.  Sections cited below are that page's "Key design" items:
 *   design 1  -- the composite implicit grid sampler I(Ax+t+Su(x)) with an
 *                implicit identity grid given by x_bounds, and its backward
 *                pass including the affine gradient;
 *   design 2  -- Mattes MI as KL(P(X,Y) || P(X)P(Y)) with the kernel density
 *                estimate P_I(v) = (1/N) sum_k kappa(v - I_k) on B bins, and
 *                LNCC from the window sums of I, J, I^2, J^2, IJ;
 *   design 5  -- the partial-aggregation identity for the MI histograms
 *                (P = sum_h (N_h/N) P^(h)), which lets callers accumulate
 *                histograms slab by slab with oracle_mi_accumulate.
 *   "Background" -- the objective L = C(F, M o phi) + R(phi) with
 *                phi(x) = Ax + t + u(x), C one of MSE, LNCC or MI, and warp
 *                composition among the memory bottlenecks: the sampler on a
 *                C-channel volume (oracle_sample_channels[_bwd], including
 *                the gradient with respect to the sampled volume) and the
 *                MSE similarity (oracle_mse).
 *
 * Readings where the page is silent (each also stated at its use):
 *   - coordinates follow the PyTorch grid_sample convention: normalised
 *     [-1, 1], align_corners=True, component order (x, y, z) = (W, H, D);
 *   - samples outside the moving image read 0 per tap (zero padding);
 *   - the trilinear slope at an integer coordinate is taken from the cell
 *     [floor(q), floor(q)+1];
 *   - u is [D][H][W][3] in normalised units of M's domain; S multiplies u;
 *     x_bounds = (x_min, x_max) are the normalised coordinates of the first
 *     and last fixed voxel along each axis;
 *   - the Parzen kernel is the cubic B-spline on both images; intensities
 *     map to bin coordinates c = 2 + (clamp(v,lo,hi)-lo)/(hi-lo)*(B-5), so
 *     every tap stays inside [0, B-1]; clamped values have zero derivative;
 *   - marginals are accumulated separately from the joint histogram;
 *   - natural log, 0*ln0 = 0, loss = -MI, N counts every fixed voxel;
 *   - LNCC is the squared local correlation cross^2/(varI*varJ+eps) built
 *     from zero-padded w^3 window sums (divisor n = w^3), averaged over all
 *     N voxels; loss = -LNCC.
 *
 * Layouts: volumes are [D][H][W] (W fastest), passed as float (fp16 inputs
 * are widened to float exactly by the caller).  dims arrays are {D, H, W}.
 * A transform is 27 doubles: A[9] (row-major, rows/cols in (x,y,z) order),
 * t[3], S[9], x_min[3], x_max[3].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* threading (OpenMP over z planes; per-plane partials merged in order) */
/* ------------------------------------------------------------------ */

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* design 1: composite implicit grid sampler                            */
/* ------------------------------------------------------------------ */

/* Identity-grid coordinate of fixed voxel i along each axis, from x_bounds:
 * x_c = x_min,c + (x_max,c - x_min,c) * i_c / (n_c - 1). */
static void fixed_coord(const double *T, const int64_t *fd, int64_t ix, int64_t iy, int64_t iz,
                        double x[3]) {
  const double *xmin = T + 21, *xmax = T + 24;
  const int64_t n[3] = {fd[2], fd[1], fd[0]};
  const int64_t i[3] = {ix, iy, iz};
  for (int c = 0; c < 3; ++c)
    x[c] = xmin[c] + (xmax[c] - xmin[c]) * (double)i[c] / (double)(n[c] - 1);
}

/* p = A x + t + S u  (normalised coordinates of the moving image). */
static void warp_point(const double *T, const double x[3], const double uv[3], double p[3]) {
  const double *A = T, *t = T + 9, *S = T + 12;
  for (int r = 0; r < 3; ++r) {
    double v = t[r];
    for (int c = 0; c < 3; ++c) v += A[r * 3 + c] * x[c];
    for (int c = 0; c < 3; ++c) v += S[r * 3 + c] * uv[c];
    p[r] = v;
  }
}

/* Value of M at integer voxel (x, y, z); 0 outside the image. */
static double m_at(const float *M, const int64_t *md, int64_t x, int64_t y, int64_t z) {
  if (x < 0 || y < 0 || z < 0 || x >= md[2] || y >= md[1] || z >= md[0]) return 0.0;
  return (double)M[(z * md[1] + y) * md[2] + x];
}

/* Trilinear value of M at normalised point p, and dJ/dp (chain through
 * q = (p+1)/2 * (n_M - 1)).  Taps outside M read 0. */
static void sample_point(const float *M, const int64_t *md, const double p[3], double *J,
                         double dJdp[3]) {
  const int64_t nM[3] = {md[2], md[1], md[0]};
  double q[3], fl[3], r[3];
  int64_t b[3];
  for (int c = 0; c < 3; ++c) {
    q[c] = (p[c] + 1.0) * 0.5 * (double)(nM[c] - 1);
    /* every tap is outside when q < -1 or q >= n: value and slope are 0 */
    if (!(q[c] >= -1.0 && q[c] < (double)nM[c])) {
      *J = 0.0;
      if (dJdp) dJdp[0] = dJdp[1] = dJdp[2] = 0.0;
      return;
    }
    fl[c] = floor(q[c]);
    b[c] = (int64_t)fl[c];
    r[c] = q[c] - fl[c];
  }
  double val = 0.0, gq[3] = {0.0, 0.0, 0.0};
  for (int cz = 0; cz < 2; ++cz)
    for (int cy = 0; cy < 2; ++cy)
      for (int cx = 0; cx < 2; ++cx) {
        const double m = m_at(M, md, b[0] + cx, b[1] + cy, b[2] + cz);
        const double wx = cx ? r[0] : 1.0 - r[0];
        const double wy = cy ? r[1] : 1.0 - r[1];
        const double wz = cz ? r[2] : 1.0 - r[2];
        val += wx * wy * wz * m;
        gq[0] += (cx ? 1.0 : -1.0) * wy * wz * m;
        gq[1] += (cy ? 1.0 : -1.0) * wx * wz * m;
        gq[2] += (cz ? 1.0 : -1.0) * wx * wy * m;
      }
  *J = val;
  if (dJdp)
    for (int c = 0; c < 3; ++c) dJdp[c] = gq[c] * 0.5 * (double)(nM[c] - 1);
}

static void load_u(const float *u, int64_t lin, double uv[3]) {
  if (u) {
    uv[0] = (double)u[lin * 3 + 0];
    uv[1] = (double)u[lin * 3 + 1];
    uv[2] = (double)u[lin * 3 + 2];
  } else {
    uv[0] = uv[1] = uv[2] = 0.0;
  }
}

/* J(x) = M(Ax + t + S u(x)) for fixed planes z0 <= z < z1.
 * J (and dJdp, [...][3], the gradient of J w.r.t. the normalised point p)
 * are indexed from plane z0.  u may be NULL (u = 0). */
void oracle_grid_sample(const float *M, const int64_t *md, const int64_t *fd, const float *u,
                        const double *T, int64_t z0, int64_t z1, double *J, double *dJdp) {
  const int64_t H = fd[1], W = fd[2];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t z = z0; z < z1; ++z)
    for (int64_t y = 0; y < H; ++y)
      for (int64_t x = 0; x < W; ++x) {
        const int64_t lin = (z * H + y) * W + x;
        const int64_t loc = ((z - z0) * H + y) * W + x;
        double xc[3], uv[3], p[3], g[3], v;
        fixed_coord(T, fd, x, y, z, xc);
        load_u(u, lin, uv);
        warp_point(T, xc, uv, p);
        sample_point(M, md, p, &v, g);
        if (J) J[loc] = v;
        if (dJdp)
          for (int c = 0; c < 3; ++c) dJdp[loc * 3 + c] = g[c];
      }
}

/* Backward of the sampler for fixed planes z0 <= z < z1, given
 * gJ = dL/dJ (indexed from plane z0):
 *   du_i = S^T (gJ_i dJ/dp_i)
 *   dA[r][c] += sum_i gJ_i dJ/dp_r x_c,   dt[r] += sum_i gJ_i dJ/dp_r.
 * du (indexed from plane z0) may be NULL.  dA and dt are ACCUMULATED into
 * (so callers can process slabs); per-plane partials are added in plane
 * order. */
void oracle_grid_sample_bwd(const float *M, const int64_t *md, const int64_t *fd, const float *u,
                            const double *T, int64_t z0, int64_t z1, const double *gJ, double *du,
                            double *dA, double *dt) {
  const int64_t H = fd[1], W = fd[2];
  const int64_t nz = z1 - z0;
  double *part = (double *)calloc((size_t)(nz > 0 ? nz : 1) * 12, sizeof(double));
  const double *S = T + 12;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t z = z0; z < z1; ++z) {
    double *pp = part + (z - z0) * 12;
    for (int64_t y = 0; y < H; ++y)
      for (int64_t x = 0; x < W; ++x) {
        const int64_t lin = (z * H + y) * W + x;
        const int64_t loc = ((z - z0) * H + y) * W + x;
        double xc[3], uv[3], p[3], g[3], v;
        fixed_coord(T, fd, x, y, z, xc);
        load_u(u, lin, uv);
        warp_point(T, xc, uv, p);
        sample_point(M, md, p, &v, g);
        const double gj = gJ[loc];
        double e[3];
        for (int r = 0; r < 3; ++r) e[r] = gj * g[r];
        if (du)
          for (int c = 0; c < 3; ++c)
            du[loc * 3 + c] = S[0 * 3 + c] * e[0] + S[1 * 3 + c] * e[1] + S[2 * 3 + c] * e[2];
        for (int r = 0; r < 3; ++r) {
          for (int c = 0; c < 3; ++c) pp[r * 3 + c] += e[r] * xc[c];
          pp[9 + r] += e[r];
        }
      }
  }
  for (int64_t z = 0; z < nz; ++z) {
    for (int k = 0; k < 9; ++k) dA[k] += part[z * 12 + k];
    for (int k = 0; k < 3; ++k) dt[k] += part[z * 12 + 9 + k];
  }
  free(part);
}

/* ------------------------------------------------------------------ */
/* design 2: Mattes mutual information with a Parzen window             */
/* ------------------------------------------------------------------ */

/* Parzen kernel.  degree 3: the cubic B-spline
 *   beta(s) = 2/3 - s^2 + |s|^3/2   (|s| < 1)
 *           = (2 - |s|)^3 / 6       (1 <= |s| < 2)
 *           = 0                     otherwise.
 * degree 0: the unit box on [-1/2, 1/2) (used only to pin the histogram
 * and entropy code: with it the joint histogram of (F, F) is diagonal). */
double oracle_bspline(int degree, double s) {
  if (degree == 0) return (s >= -0.5 && s < 0.5) ? 1.0 : 0.0;
  const double a = fabs(s);
  if (a < 1.0) return 2.0 / 3.0 - a * a + 0.5 * a * a * a;
  if (a < 2.0) {
    const double b = 2.0 - a;
    return b * b * b / 6.0;
  }
  return 0.0;
}

/* d beta / d s for the cubic B-spline (0 for the box). */
double oracle_bspline_deriv(int degree, double s) {
  if (degree == 0) return 0.0;
  const double a = fabs(s);
  const double sg = s < 0.0 ? -1.0 : 1.0;
  if (a < 1.0) return sg * (-2.0 * a + 1.5 * a * a);
  if (a < 2.0) {
    const double b = 2.0 - a;
    return -sg * 0.5 * b * b;
  }
  return 0.0;
}

/* Bin coordinate of intensity v: c = 2 + (clamp(v,lo,hi) - lo)/(hi - lo) * (B - 5),
 * so c lies in [2, B-3] and the kernel taps stay in [0, B-1].
 * *dcdv = (B-5)/(hi-lo) when lo <= v <= hi, else 0 (clamped). */
double oracle_bin_coord(double v, double lo, double hi, int B, double *dcdv) {
  double cv = v, d = (double)(B - 5) / (hi - lo);
  if (v < lo) {
    cv = lo;
    d = 0.0;
  } else if (v > hi) {
    cv = hi;
    d = 0.0;
  }
  if (dcdv) *dcdv = d;
  return 2.0 + (cv - lo) / (hi - lo) * (double)(B - 5);
}

/* Lowest bin the kernel can touch for bin coordinate c. */
static int first_tap(int degree, double c) { return degree == 0 ? (int)floor(c + 0.5) : (int)floor(c) - 1; }
static int n_taps(int degree) { return degree == 0 ? 1 : 4; }

/* Un-normalised Parzen histograms over n voxels, ACCUMULATED into
 *   H[a*B+b] += sum_k beta(a - cF_k) beta(b - cJ_k),
 *   HF[a]    += sum_k beta(a - cF_k),   HJ[b] += sum_k beta(b - cJ_k).
 * Bins outside a voxel's taps get exactly beta = 0, so only the taps are
 * visited.  Per-thread partials are merged in thread order. */
void oracle_mi_accumulate(const float *F, const double *J, int64_t n, int B, int degree, double flo,
                          double fhi, double jlo, double jhi, double *H, double *HF, double *HJ) {
  const int nt = oracle_max_threads();
  const size_t per = (size_t)B * B + 2 * (size_t)B;
  double *loc = (double *)calloc((size_t)nt * per, sizeof(double));
#pragma omp parallel
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double *h = loc + (size_t)tid * per, *hf = h + (size_t)B * B, *hj = hf + B;
#pragma omp for schedule(static)
    for (int64_t k = 0; k < n; ++k) {
      const double cf = oracle_bin_coord((double)F[k], flo, fhi, B, NULL);
      const double cj = oracle_bin_coord(J[k], jlo, jhi, B, NULL);
      const int a0 = first_tap(degree, cf), b0 = first_tap(degree, cj), nk = n_taps(degree);
      for (int ia = 0; ia < nk; ++ia) {
        const int a = a0 + ia;
        const double wa = oracle_bspline(degree, (double)a - cf);
        hf[a] += wa;
        for (int ib = 0; ib < nk; ++ib) {
          const int b = b0 + ib;
          h[a * B + b] += wa * oracle_bspline(degree, (double)b - cj);
        }
      }
      for (int ib = 0; ib < nk; ++ib) {
        const int b = b0 + ib;
        hj[b] += oracle_bspline(degree, (double)b - cj);
      }
    }
  }
  for (int t = 0; t < nt; ++t) {
    const double *h = loc + (size_t)t * per;
    for (size_t i = 0; i < (size_t)B * B; ++i) H[i] += h[i];
    for (int i = 0; i < B; ++i) HF[i] += h[(size_t)B * B + i];
    for (int i = 0; i < B; ++i) HJ[i] += h[(size_t)B * B + B + i];
  }
  free(loc);
}

/* Normalise by N (P = H/N etc.) and return
 *   MI = sum_{P(a,b) > 0} P(a,b) [ln P(a,b) - ln P_F(a) - ln P_J(b)].
 * P, PF, PJ may alias H, HF, HJ. */
double oracle_mi_finish(const double *H, const double *HF, const double *HJ, int B, double N,
                        double *P, double *PF, double *PJ) {
  for (int i = 0; i < B * B; ++i) P[i] = H[i] / N;
  for (int i = 0; i < B; ++i) {
    PF[i] = HF[i] / N;
    PJ[i] = HJ[i] / N;
  }
  double mi = 0.0;
  for (int a = 0; a < B; ++a)
    for (int b = 0; b < B; ++b) {
      const double p = P[a * B + b];
      if (p > 0.0) mi += p * (log(p) - log(PF[a]) - log(PJ[b]));
    }
  return mi;
}

/* Gradient of the loss -MI with respect to J_k, by the full chain rule
 * through the joint P and the moving marginal P_J (P_F does not depend on J):
 *   dMI/dJ_k = sum_{a,b} (ln P - ln P_F - ln P_J + 1) dP(a,b)/dJ_k
 *            - sum_b (sum_a P(a,b) / P_J(b)) dP_J(b)/dJ_k,
 *   dP(a,b)/dJ_k = -(c'_k/N) beta(a - cF_k) beta'(b - cJ_k),
 *   dP_J(b)/dJ_k = -(c'_k/N) beta'(b - cJ_k).
 * No term is dropped even where it cancels analytically.  Cubic only. */
void oracle_mi_grad(const float *F, const double *J, int64_t n, int B, double flo, double fhi,
                    double jlo, double jhi, const double *P, const double *PF, const double *PJ,
                    double N, double *dJ) {
  double *colsum = (double *)calloc((size_t)B, sizeof(double));
  for (int b = 0; b < B; ++b)
    for (int a = 0; a < B; ++a) colsum[b] += P[a * B + b];
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < n; ++k) {
    double dc;
    const double cf = oracle_bin_coord((double)F[k], flo, fhi, B, NULL);
    const double cj = oracle_bin_coord(J[k], jlo, jhi, B, &dc);
    const int a0 = (int)floor(cf) - 1, b0 = (int)floor(cj) - 1;
    double g = 0.0;
    for (int ib = 0; ib < 4; ++ib) {
      const int b = b0 + ib;
      const double dbeta = oracle_bspline_deriv(3, (double)b - cj);
      const double dPJ = -(dc / N) * dbeta;
      for (int ia = 0; ia < 4; ++ia) {
        const int a = a0 + ia;
        const double p = P[a * B + b];
        const double dP = -(dc / N) * oracle_bspline(3, (double)a - cf) * dbeta;
        if (p > 0.0) g += (log(p) - log(PF[a]) - log(PJ[b]) + 1.0) * dP;
      }
      if (PJ[b] > 0.0) g -= (colsum[b] / PJ[b]) * dPJ;
    }
    dJ[k] = -g;
  }
  free(colsum);
}

/* Convenience: MI over n voxels (accumulate, finish), optional gradient of
 * -MI into dJ.  P is B*B, PF and PJ are B (outputs, normalised). */
double oracle_mi(const float *F, const double *J, int64_t n, int B, int degree, double flo,
                 double fhi, double jlo, double jhi, double *P, double *PF, double *PJ, double *dJ) {
  memset(P, 0, sizeof(double) * (size_t)B * B);
  memset(PF, 0, sizeof(double) * (size_t)B);
  memset(PJ, 0, sizeof(double) * (size_t)B);
  oracle_mi_accumulate(F, J, n, B, degree, flo, fhi, jlo, jhi, P, PF, PJ);
  const double mi = oracle_mi_finish(P, PF, PJ, B, (double)n, P, PF, PJ);
  if (dJ && degree == 3) oracle_mi_grad(F, J, n, B, flo, fhi, jlo, jhi, P, PF, PJ, (double)n, dJ);
  return mi;
}

/* ------------------------------------------------------------------ */
/* design 2: local normalised cross correlation                         */
/* ------------------------------------------------------------------ */

/* LNCC of F and J on a [D][H][W] grid with an odd window w (r = (w-1)/2,
 * n = w^3), zero padding:
 *   S_X(k)  = sum_{m in cube(k,r), m inside the grid} X_m, X in {F, J, F^2, J^2, FJ}
 *   cross   = S_FJ - S_F S_J / n,  vF = S_FF - S_F^2/n,  vJ = S_JJ - S_J^2/n
 *   cc_k    = cross^2 / (vF vJ + eps),   LNCC = (1/N) sum_k cc_k.
 * Returns LNCC.  cc (N) is optional.  dJ (N, optional) receives the gradient
 * of the loss -LNCC:
 *   D = vF vJ + eps
 *   g_FJ(k) = -(1/N) 2 cross / D
 *   g_JJ(k) = -(1/N) (-cross^2 vF / D^2)
 *   g_J(k)  = -(1/N) [ -(2 cross / D) S_F / n + (cross^2 vF / D^2)(2 S_J / n) ]
 *   dJ_m    = sum_{k in cube(m,r), k inside} g_J(k) + 2 J_m g_JJ(k) + F_m g_FJ(k). */
double oracle_lncc(const float *F, const double *J, const int64_t *dims, int w, double eps,
                   double *cc, double *dJ) {
  const int64_t D = dims[0], H = dims[1], W = dims[2];
  const int64_t N = D * H * W;
  const int r = (w - 1) / 2;
  const double n = (double)w * w * w;
  double *gam = dJ ? (double *)malloc(sizeof(double) * 3 * (size_t)N) : NULL;
  double *plane = (double *)calloc((size_t)D, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t z = 0; z < D; ++z)
    for (int64_t y = 0; y < H; ++y)
      for (int64_t x = 0; x < W; ++x) {
        double sF = 0, sJ = 0, sFF = 0, sJJ = 0, sFJ = 0;
        for (int64_t zz = z - r; zz <= z + r; ++zz) {
          if (zz < 0 || zz >= D) continue;
          for (int64_t yy = y - r; yy <= y + r; ++yy) {
            if (yy < 0 || yy >= H) continue;
            for (int64_t xx = x - r; xx <= x + r; ++xx) {
              if (xx < 0 || xx >= W) continue;
              const int64_t m = (zz * H + yy) * W + xx;
              const double f = (double)F[m], j = J[m];
              sF += f;
              sJ += j;
              sFF += f * f;
              sJJ += j * j;
              sFJ += f * j;
            }
          }
        }
        const double cross = sFJ - sF * sJ / n;
        const double vF = sFF - sF * sF / n;
        const double vJ = sJJ - sJ * sJ / n;
        const double Dn = vF * vJ + eps;
        const double c = cross * cross / Dn;
        const int64_t k = (z * H + y) * W + x;
        if (cc) cc[k] = c;
        plane[z] += c;
        if (gam) {
          gam[3 * k + 0] = -(1.0 / (double)N) * (-(2.0 * cross / Dn) * sF / n +
                                                  (cross * cross * vF / (Dn * Dn)) * (2.0 * sJ / n));
          gam[3 * k + 1] = -(1.0 / (double)N) * (-cross * cross * vF / (Dn * Dn));
          gam[3 * k + 2] = -(1.0 / (double)N) * (2.0 * cross / Dn);
        }
      }
  double tot = 0.0;
  for (int64_t z = 0; z < D; ++z) tot += plane[z];
  free(plane);
  if (gam) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t z = 0; z < D; ++z)
      for (int64_t y = 0; y < H; ++y)
        for (int64_t x = 0; x < W; ++x) {
          const int64_t m = (z * H + y) * W + x;
          double gJ = 0, gJJ = 0, gFJ = 0;
          for (int64_t zz = z - r; zz <= z + r; ++zz) {
            if (zz < 0 || zz >= D) continue;
            for (int64_t yy = y - r; yy <= y + r; ++yy) {
              if (yy < 0 || yy >= H) continue;
              for (int64_t xx = x - r; xx <= x + r; ++xx) {
                if (xx < 0 || xx >= W) continue;
                const int64_t k = (zz * H + yy) * W + xx;
                gJ += gam[3 * k + 0];
                gJJ += gam[3 * k + 1];
                gFJ += gam[3 * k + 2];
              }
            }
          }
          dJ[m] = gJ + 2.0 * J[m] * gJJ + (double)F[m] * gFJ;
        }
    free(gam);
  }
  return tot / (double)N;
}

/* ------------------------------------------------------------------ */
/* warp composition: the design-1 sampler on a C-channel volume         */
/* ------------------------------------------------------------------ */

/* The "Background" section names deformation interpolation and warp
 * composition as the first of the three memory bottlenecks; design 1's
 * sampler I(Ax + t + Su(x)) applies unchanged when I has several channels.
 * A channel-last volume V is [Dv][Hv][Wv][C] (channel fastest).  Composing a
 * displacement field V (C = 3, normalised units of its own domain) after
 * phi(x) = Ax + t + Su(x) gives
 *   V o phi composed:  phi_V(phi(x)) = phi(x) + V(phi(x)) = Ax + t + d(x),
 *   d(x) = S u(x) + V(phi(x)),
 * i.e. the composite warp in the same form with S = I and displacement d.
 * Readings: the same conventions as the scalar sampler (align_corners grid,
 * zero padding per tap, floor cell for the slope); `compose` adds S u(x). */

/* Value of channel ch of V at integer voxel (x, y, z); 0 outside. */
static double v_at(const float *V, int C, const int64_t *vd, int64_t x, int64_t y, int64_t z, int ch) {
  if (x < 0 || y < 0 || z < 0 || x >= vd[2] || y >= vd[1] || z >= vd[0]) return 0.0;
  return (double)V[((z * vd[1] + y) * vd[2] + x) * C + ch];
}

/* Cell of normalised point p in a volume of extents vd: corner b, fractions
 * r; returns 0 when every tap is outside (q < -1 or q >= n on some axis). */
static int cell_of_point(const int64_t *vd, const double p[3], int64_t b[3], double r[3]) {
  const int64_t n[3] = {vd[2], vd[1], vd[0]};
  for (int c = 0; c < 3; ++c) {
    const double q = (p[c] + 1.0) * 0.5 * (double)(n[c] - 1);
    if (!(q >= -1.0 && q < (double)n[c])) return 0;
    const double fl = floor(q);
    b[c] = (int64_t)fl;
    r[c] = q - fl;
  }
  return 1;
}

/* Trilinear weight of corner (cx, cy, cz) of a cell with fractions r. */
static double corner_weight(const double r[3], int cx, int cy, int cz) {
  return (cx ? r[0] : 1.0 - r[0]) * (cy ? r[1] : 1.0 - r[1]) * (cz ? r[2] : 1.0 - r[2]);
}

/* Sampled channels val[C] at p and their slopes dvdp[C][3] w.r.t. p. */
static void sample_channels_point(const float *V, int C, const int64_t *vd, const double p[3], double *val,
                                  double *dvdp) {
  const int64_t n[3] = {vd[2], vd[1], vd[0]};
  int64_t b[3];
  double r[3];
  for (int ch = 0; ch < C; ++ch) {
    val[ch] = 0.0;
    if (dvdp) dvdp[ch * 3 + 0] = dvdp[ch * 3 + 1] = dvdp[ch * 3 + 2] = 0.0;
  }
  if (!cell_of_point(vd, p, b, r)) return;
  for (int cz = 0; cz < 2; ++cz)
    for (int cy = 0; cy < 2; ++cy)
      for (int cx = 0; cx < 2; ++cx) {
        const double wx = cx ? r[0] : 1.0 - r[0];
        const double wy = cy ? r[1] : 1.0 - r[1];
        const double wz = cz ? r[2] : 1.0 - r[2];
        for (int ch = 0; ch < C; ++ch) {
          const double m = v_at(V, C, vd, b[0] + cx, b[1] + cy, b[2] + cz, ch);
          val[ch] += wx * wy * wz * m;
          if (dvdp) {
            dvdp[ch * 3 + 0] += (cx ? 1.0 : -1.0) * wy * wz * m * 0.5 * (double)(n[0] - 1);
            dvdp[ch * 3 + 1] += (cy ? 1.0 : -1.0) * wx * wz * m * 0.5 * (double)(n[1] - 1);
            dvdp[ch * 3 + 2] += (cz ? 1.0 : -1.0) * wx * wy * m * 0.5 * (double)(n[2] - 1);
          }
        }
      }
}

/* out[i][c] = V_c(A x_i + t + S u_i) (+ (S u_i)_c when compose, C = 3) for
 * fixed planes z0 <= z < z1; out is [z1-z0][H][W][C], indexed from z0. */
void oracle_sample_channels(const float *V, int C, const int64_t *vd, const int64_t *fd, const float *u,
                            const double *T, int compose, int64_t z0, int64_t z1, double *out) {
  const int64_t H = fd[1], W = fd[2];
  const double *S = T + 12;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t z = z0; z < z1; ++z)
    for (int64_t y = 0; y < H; ++y)
      for (int64_t x = 0; x < W; ++x) {
        const int64_t lin = (z * H + y) * W + x;
        const int64_t loc = ((z - z0) * H + y) * W + x;
        double xc[3], uv[3], p[3], val[4];
        fixed_coord(T, fd, x, y, z, xc);
        load_u(u, lin, uv);
        warp_point(T, xc, uv, p);
        sample_channels_point(V, C, vd, p, val, NULL);
        for (int ch = 0; ch < C; ++ch) {
          double v = val[ch];
          if (compose) v += S[ch * 3 + 0] * uv[0] + S[ch * 3 + 1] * uv[1] + S[ch * 3 + 2] * uv[2];
          out[loc * C + ch] = v;
        }
      }
}

/* Backward of oracle_sample_channels for planes z0 <= z < z1 given
 * gout = dL/dout ([z1-z0][H][W][C]):
 *   e_i      = sum_c gout_ic dV_c/dp (p_i)
 *   du_i     = S^T e_i  (+ S^T gout_i when compose)
 *   dA[r][c] += sum_i e_ir x_ic,   dt[r] += sum_i e_ir
 *   dV[v][c] += sum_i gout_ic w_v(p_i)   (w_v: trilinear weight of corner v)
 * du (indexed from z0) and dV may be NULL; dA, dt and dV are ACCUMULATED
 * (per-plane partials of dA, dt added in plane order).  With dV the planes
 * run serially (the scatter has no fixed owner per voxel); without it,
 * OpenMP over planes. */
static void channels_bwd_plane(const float *V, int C, const int64_t *vd, const int64_t *fd, const float *u,
                               const double *T, int compose, int64_t z0, int64_t z, const double *gout,
                               double *du, double *pp, double *dV) {
  const int64_t H = fd[1], W = fd[2];
  const double *S = T + 12;
  for (int64_t y = 0; y < H; ++y)
    for (int64_t x = 0; x < W; ++x) {
      const int64_t lin = (z * H + y) * W + x;
      const int64_t loc = ((z - z0) * H + y) * W + x;
      double xc[3], uv[3], p[3], val[4], dv[12], e[3] = {0.0, 0.0, 0.0};
      fixed_coord(T, fd, x, y, z, xc);
      load_u(u, lin, uv);
      warp_point(T, xc, uv, p);
      sample_channels_point(V, C, vd, p, val, dv);
      const double *g = gout + loc * C;
      for (int ch = 0; ch < C; ++ch)
        for (int r = 0; r < 3; ++r) e[r] += g[ch] * dv[ch * 3 + r];
      if (du)
        for (int c = 0; c < 3; ++c) {
          double s = S[0 * 3 + c] * e[0] + S[1 * 3 + c] * e[1] + S[2 * 3 + c] * e[2];
          if (compose) s += S[0 * 3 + c] * g[0] + S[1 * 3 + c] * g[1] + S[2 * 3 + c] * g[2];
          du[loc * 3 + c] = s;
        }
      for (int r = 0; r < 3; ++r) {
        for (int c = 0; c < 3; ++c) pp[r * 3 + c] += e[r] * xc[c];
        pp[9 + r] += e[r];
      }
      if (dV) {
        int64_t b[3];
        double rr[3];
        if (!cell_of_point(vd, p, b, rr)) continue;
        for (int cz = 0; cz < 2; ++cz)
          for (int cy = 0; cy < 2; ++cy)
            for (int cx = 0; cx < 2; ++cx) {
              const int64_t vx = b[0] + cx, vy = b[1] + cy, vz = b[2] + cz;
              if (vx < 0 || vy < 0 || vz < 0 || vx >= vd[2] || vy >= vd[1] || vz >= vd[0]) continue;
              const double w = corner_weight(rr, cx, cy, cz);
              const int64_t v = (vz * vd[1] + vy) * vd[2] + vx;
              for (int ch = 0; ch < C; ++ch) dV[v * C + ch] += g[ch] * w;
            }
      }
    }
}

void oracle_sample_channels_bwd(const float *V, int C, const int64_t *vd, const int64_t *fd, const float *u,
                                const double *T, int compose, int64_t z0, int64_t z1, const double *gout,
                                double *du, double *dA, double *dt, double *dV) {
  const int64_t nz = z1 - z0;
  double *part = (double *)calloc((size_t)(nz > 0 ? nz : 1) * 12, sizeof(double));
  if (dV) {
    for (int64_t z = z0; z < z1; ++z)
      channels_bwd_plane(V, C, vd, fd, u, T, compose, z0, z, gout, du, part + (z - z0) * 12, dV);
  } else {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t z = z0; z < z1; ++z)
      channels_bwd_plane(V, C, vd, fd, u, T, compose, z0, z, gout, du, part + (z - z0) * 12, NULL);
  }
  for (int64_t z = 0; z < nz; ++z) {
    for (int k = 0; k < 9; ++k) dA[k] += part[z * 12 + k];
    for (int k = 0; k < 3; ++k) dt[k] += part[z * 12 + 9 + k];
  }
  free(part);
}

/* ------------------------------------------------------------------ */
/* MSE similarity                                                       */
/* ------------------------------------------------------------------ */

/* "Background": C(F, M o phi) may be the mean squared error; design 5 calls
 * it a per-voxel loss.  MSE = (1/n) sum_k (J_k - F_k)^2 and
 * dMSE/dJ_k = 2 (J_k - F_k) / n (dJ may be NULL).  Plain sum in index
 * order. */
double oracle_mse(const float *F, const double *J, int64_t n, double *dJ) {
  double s = 0.0;
  for (int64_t k = 0; k < n; ++k) {
    const double d = J[k] - (double)F[k];
    s += d * d;
    if (dJ) dJ[k] = 2.0 * d / (double)n;
  }
  return s / (double)n;
}

/* ------------------------------------------------------------------ */
/* Sobolev regulariser and the Adam update of the displacement field    */
/* ------------------------------------------------------------------ */

/* "Background": L(phi) = C(F, M o phi) + R(phi) with R a Sobolev norm; the
 * overview updates the warp shards by gradient descent with optimiser state
 * [m1], [m2] held per voxel beside u.  Readings (the page gives no formula):
 *   R(u) = (lambda / N) sum_c sum_a sum_{i : i + e_a inside} (u_c(i + e_a) - u_c(i))^2,
 * the first-order Sobolev (H^1) seminorm of u with forward differences in
 * voxel units and no term across the boundary; its gradient is
 *   dR/du_c(i) = (2 lambda / N) sum_{j neighbour of i inside} (u_c(i) - u_c(j)).
 * u is [D][H][W][3].  dR may be NULL. */
double oracle_sobolev(const float *u, const int64_t *fd, double lambda, double *dR) {
  const int64_t D = fd[0], H = fd[1], W = fd[2];
  const double N = (double)(D * H * W);
  double *plane = (double *)calloc((size_t)D, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t z = 0; z < D; ++z) {
    double s = 0.0;
    for (int64_t y = 0; y < H; ++y)
      for (int64_t x = 0; x < W; ++x) {
        const int64_t i = (z * H + y) * W + x;
        const int64_t nb[6][3] = {{x + 1, y, z}, {x, y + 1, z}, {x, y, z + 1},
                                  {x - 1, y, z}, {x, y - 1, z}, {x, y, z - 1}};
        double g[3] = {0.0, 0.0, 0.0};
        for (int k = 0; k < 6; ++k) {
          const int64_t xx = nb[k][0], yy = nb[k][1], zz = nb[k][2];
          if (xx < 0 || yy < 0 || zz < 0 || xx >= W || yy >= H || zz >= D) continue;
          const int64_t j = (zz * H + yy) * W + xx;
          for (int c = 0; c < 3; ++c) {
            const double d = (double)u[3 * j + c] - (double)u[3 * i + c];
            if (k < 3) s += d * d;  /* forward edges: each edge once */
            g[c] -= d;              /* u_i - u_j summed over neighbours */
          }
        }
        if (dR)
          for (int c = 0; c < 3; ++c) dR[3 * i + c] = 2.0 * lambda / N * g[c];
      }
    plane[z] = s;
  }
  double tot = 0.0;
  for (int64_t z = 0; z < D; ++z) tot += plane[z];
  free(plane);
  return lambda / N * tot;
}

/* One Adam step (Kingma & Ba, with bias correction) on n values, step t >= 1:
 *   m1 = b1 m1 + (1 - b1) g,   m2 = b2 m2 + (1 - b2) g^2,
 *   x -= lr (m1 / (1 - b1^t)) / (sqrt(m2 / (1 - b2^t)) + eps).
 * x, m1, m2 are updated in place. */
void oracle_adam(double *x, const double *g, double *m1, double *m2, int64_t n, double lr, double b1, double b2,
                 double eps, int t) {
  const double c1 = 1.0 - pow(b1, (double)t), c2 = 1.0 - pow(b2, (double)t);
  for (int64_t k = 0; k < n; ++k) {
    m1[k] = b1 * m1[k] + (1.0 - b1) * g[k];
    m2[k] = b2 * m2[k] + (1.0 - b2) * g[k] * g[k];
    x[k] -= lr * (m1[k] / c1) / (sqrt(m2[k] / c2) + eps);
  }
}
