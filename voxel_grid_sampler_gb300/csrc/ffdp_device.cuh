// ffdp_device.cuh -- device building blocks shared by the libffdp kernels.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration", Key designs item 1 (coordinates of I(Ax+t+Su(x)) computed in
// registers from x_bounds; nothing grid-sized is materialised) and item 2
// (Parzen-window MI with a shared-memory histogram; LNCC window sums).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ffdp {

// ---------------------------------------------------------------- constants
#ifndef FFDP_SWEEP1_THREADS
#define FFDP_SWEEP1_THREADS 640
#endif
#ifndef FFDP_SWEEP2_THREADS
#define FFDP_SWEEP2_THREADS 512
#endif
#ifndef FFDP_SWEEP2_STREAM_THREADS
#define FFDP_SWEEP2_STREAM_THREADS 768
#endif
// threads per CTA (one CTA per SM) of the histogram / forward sweep, of the
// gradient sweep that gathers M again (more registers per thread), and of the
// gradient sweeps that only stream stored per-voxel inputs (more warps keep
// more bulk copies and stores in flight)
constexpr int kSweep1Threads = FFDP_SWEEP1_THREADS;
constexpr int kSweep2Threads = FFDP_SWEEP2_THREADS;
constexpr int kSweep2StreamThreads = FFDP_SWEEP2_STREAM_THREADS;
constexpr int kVPT = 4;                 // voxels per sweep thread per iteration (32 apart)
constexpr int kHistFrac = 20;           // fixed-point fraction bits of histogram weights
constexpr float kHistOne = 1048576.0f;  // 2^kHistFrac
// histogram weight scales whose product is 2^(kHistFrac - 149): a product of
// two weights is then the subnormal float holding the fixed-point count
constexpr float kHistScaleF = 2.7105054312137611e-20f;  // 2^-65
constexpr float kHistScaleJ = 5.4210108624275222e-20f;  // 2^-64
static_assert(kHistFrac == 20, "kHistScaleF * kHistScaleJ = 2^(kHistFrac - 149)");
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: x + kMagic holds round(x) in its low bits
constexpr unsigned kMagicBits = 0x4B400000u;
constexpr int kPartialStride = 16;      // doubles per CTA partial record

// Per-CTA partial record layout (doubles), reduced by the finish kernel:
//   [0..2]  s_r   = sum g dJ/dq_r
//   [3..11] m_rc  = sum g dJ/dq_r (i_c - c_c)   (c_c: grid centre index)
//   [12]    sum cc (LNCC)
//   [13]    sum (J - F)^2 (MSE)
enum { kPS = 0, kPM = 3, kPCC = 12, kPSE = 13 };

// ------------------------------------------------------------ geometry
// Fixed-grid index i = (ix, iy, iz) maps to moving-image voxel coordinates
//   q = G i + g0 + K u,   G = diag(hM) A diag(dx),  g0 = hM (A x_min + t + 1),
//   K = diag(hM) S,       hM = (n_M - 1)/2,          dx = (x_max - x_min)/(n_F - 1).
// G i + g0 is carried in 64-bit fixed point with 32 fraction bits, so the
// integer cell index and the in-cell fraction stay exact to ~1e-7 voxel even
// on 1024^3 grids (a float32 q would round at 6e-5 voxel there).
struct Geom {
  long long Gq[9];  // [r][c], 2^-32 units
  long long g0q[3];
  float Gx[3];      // G[r][0]: q step per fixed voxel along x (float)
  float K[9];       // [r][c]
  float hM[3];
  float ctr[3];     // grid centre index (n_F - 1)/2 per axis (x, y, z)
  int fW, fH, fD;   // fixed grid extents
  int mW, mH, mD;   // moving grid extents
  long long mHW;
  unsigned N;       // fixed voxels
  unsigned divW_m, divHW_m;  // fast division magic numbers for W and H*W
  int divW_s, divHW_s;
  int k_diag;       // K is diagonal (S diagonal): u enters q component-wise
  int a_diag;       // G is diagonal (A diagonal)
  int ia;           // G = I and g0 integer: every anchor is the integer i + io
  int io[3];        // g0 when ia
};

// Unsigned division by a runtime-invariant divisor (round-up method).
__device__ __forceinline__ unsigned fast_div(unsigned n, unsigned m, int s) {
  return (unsigned)(((unsigned long long)__umulhi(n, m) + n) >> s);
}

__device__ __forceinline__ void lin_to_xyz(const Geom& g, unsigned lin, int& ix, int& iy, int& iz) {
  unsigned z = fast_div(lin, g.divHW_m, g.divHW_s);
  unsigned rem = lin - z * ((unsigned)g.fW * (unsigned)g.fH);
  unsigned y = fast_div(rem, g.divW_m, g.divW_s);
  iz = (int)z;
  iy = (int)y;
  ix = (int)(rem - y * (unsigned)g.fW);
}

// 64-bit fixed-point anchor P = G i + g0 (no displacement).
__device__ __forceinline__ void anchor(const Geom& g, int ix, int iy, int iz, long long P[3]) {
  if (g.a_diag) {
    P[0] = g.g0q[0] + g.Gq[0] * ix;
    P[1] = g.g0q[1] + g.Gq[4] * iy;
    P[2] = g.g0q[2] + g.Gq[8] * iz;
  } else {
#pragma unroll
    for (int r = 0; r < 3; ++r)
      P[r] = g.g0q[r] + g.Gq[r * 3 + 0] * ix + g.Gq[r * 3 + 1] * iy + g.Gq[r * 3 + 2] * iz;
  }
}

// floor(t) and t - floor(t) for |t| < 2^21 with full-rate float/int ops:
// x + 1.5*2^23 rounds to the nearest integer, corrected by one when it
// rounded up.
__device__ __forceinline__ void floor_split(float t, int& fi, float& fr) {
#ifndef FFDP_FLOOR_MAGIC_ONLY
  // round-down instruction, then the exact integer through the same trick
  const float fl = floorf(t);
  fi = (int)(__float_as_uint(fl + kMagic) - kMagicBits);
  fr = t - fl;
#else
  float a = t + kMagic;
  float fl = a - kMagic;
  int i = (int)(__float_as_uint(a) - kMagicBits);
  if (fl > t) {
    fl -= 1.0f;
    i -= 1;
  }
  fi = i;
  fr = t - fl;
#endif
}

// Cell of the moving image containing q = P + K u: integer corner b and
// fractions r.  The in-cell coordinate is clamped to +-2^20, so |b| < 2^26
// (|k| < 2^25 by the host-side range check) and every consumer's unsigned
// range test rejects far-away corners without overflow.
__device__ __forceinline__ void cell_of(const Geom& g, const long long P[3], float u0, float u1,
                                        float u2, int b[3], float r[3]) {
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    const int k = (int)(P[c] >> 32);
    const unsigned lo = (unsigned)(P[c] & 0xffffffffll);
    const float f = __uint_as_float(0x3f800000u | (lo >> 9)) - 1.0f;  // [0, 1)
    float t;
    if (g.k_diag) {
      t = fmaf(g.K[c * 4], c == 0 ? u0 : (c == 1 ? u1 : u2), f);
    } else {
      t = fmaf(g.K[c * 3 + 0], u0, fmaf(g.K[c * 3 + 1], u1, fmaf(g.K[c * 3 + 2], u2, f)));
    }
    t = fminf(fmaxf(t, -1048576.0f), 1048576.0f);
    int fi;
    float fr;
    floor_split(t, fi, fr);
    b[c] = k + fi;
    r[c] = fr;
  }
}

// The same cell when every anchor is an integer (G = I, g0 = io integer: a
// grid sampled at its own voxel positions up to an integer shift, as for
// A = I, t = 0 and equal fixed and moving extents): the fraction of the
// anchor is 0, so q = (i + io) + K u with no fixed-point arithmetic.  Gives
// the same b and r as cell_of on such anchors.
__device__ __forceinline__ void cell_of_int(const Geom& g, int ix, int iy, int iz, float u0, float u1, float u2,
                                            int b[3], float r[3]) {
  const int idx[3] = {ix, iy, iz};
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    float t;
    if (g.k_diag) {
      t = g.K[c * 4] * (c == 0 ? u0 : (c == 1 ? u1 : u2));
    } else {
      t = fmaf(g.K[c * 3 + 0], u0, fmaf(g.K[c * 3 + 1], u1, g.K[c * 3 + 2] * u2));
    }
    t = fminf(fmaxf(t, -1048576.0f), 1048576.0f);
    int fi;
    float fr;
    floor_split(t, fi, fr);
    b[c] = idx[c] + g.io[c] + fi;
    r[c] = fr;
  }
}

// ------------------------------------------------- packed fp32 pairs
// Blackwell executes add/sub/mul/fma on a pair of fp32 values held in a
// 64-bit register pair as one instruction (PTX .f32x2, sm_100 and later).
__device__ __forceinline__ unsigned long long f2_bits(float2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 bits_f2(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}

// ------------------------------------------------------------- M access
// Raw tap registers: a float register holds either an fp32 tap or the 16
// bits of an fp16 tap.  Half taps are converted only when they are
// interpolated, so no conversion sits between the loads of a cell and the
// eight loads stay in flight together.
template <typename T>
__device__ __forceinline__ float ldg_raw(const T* p);
template <>
__device__ __forceinline__ float ldg_raw<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float ldg_raw<__half>(const __half* p) {
  return __uint_as_float((unsigned)__ldg(reinterpret_cast<const unsigned short*>(p)));
}
template <typename T>
__device__ __forceinline__ float tap_value(float raw);
template <>
__device__ __forceinline__ float tap_value<float>(float raw) {
  return raw;
}
template <>
__device__ __forceinline__ float tap_value<__half>(float raw) {
  return __half2float(__ushort_as_half((unsigned short)__float_as_uint(raw)));
}

// The 8 raw taps of cell b (m[z][y][x] order: 000,001,010,011,100,101,110,111),
// zero outside M (the zero bit pattern is +0 in both types).  Split from the
// interpolation so callers can issue the loads of several voxels before
// using any of them.
template <typename MT>
__device__ __forceinline__ void gather8(const MT* __restrict__ M, const Geom& g, const int b[3], float m[8]) {
  const int bx = b[0], by = b[1], bz = b[2];
  if ((unsigned)bx < (unsigned)(g.mW - 1) && (unsigned)by < (unsigned)(g.mH - 1) &&
      (unsigned)bz < (unsigned)(g.mD - 1)) {
    const unsigned off = ((unsigned)bz * (unsigned)g.mH + (unsigned)by) * (unsigned)g.mW + (unsigned)bx;
    const MT* p = M + off;
    const MT* q = M + (off + (unsigned)g.mW);
    const MT* p2 = M + (off + (unsigned)g.mHW);
    const MT* q2 = M + (off + (unsigned)g.mHW + (unsigned)g.mW);
    m[0] = ldg_raw(p);
    m[1] = ldg_raw(p + 1);
    m[2] = ldg_raw(q);
    m[3] = ldg_raw(q + 1);
    m[4] = ldg_raw(p2);
    m[5] = ldg_raw(p2 + 1);
    m[6] = ldg_raw(q2);
    m[7] = ldg_raw(q2 + 1);
  } else {
    const bool x0 = (unsigned)bx < (unsigned)g.mW, x1 = (unsigned)(bx + 1) < (unsigned)g.mW;
    const bool y0 = (unsigned)by < (unsigned)g.mH, y1 = (unsigned)(by + 1) < (unsigned)g.mH;
    const bool z0 = (unsigned)bz < (unsigned)g.mD, z1 = (unsigned)(bz + 1) < (unsigned)g.mD;
    auto at = [&](int dz, int dy, int dx, bool ok) -> float {
      return ok ? ldg_raw(M + ((long long)(bz + dz) * g.mH + (by + dy)) * g.mW + (bx + dx)) : 0.0f;
    };
    m[0] = at(0, 0, 0, z0 && y0 && x0);
    m[1] = at(0, 0, 1, z0 && y0 && x1);
    m[2] = at(0, 1, 0, z0 && y1 && x0);
    m[3] = at(0, 1, 1, z0 && y1 && x1);
    m[4] = at(1, 0, 0, z1 && y0 && x0);
    m[5] = at(1, 0, 1, z1 && y0 && x1);
    m[6] = at(1, 1, 0, z1 && y1 && x0);
    m[7] = at(1, 1, 1, z1 && y1 && x1);
  }
}

// Trilinear value (and optionally dJ/dq) from the 8 taps and fractions r.
template <bool GRAD>
__device__ __forceinline__ float interp8(const float m[8], const float r[3], float& gx, float& gy, float& gz) {
  const float rz = r[2];
  const float2 rx2 = make_float2(r[0], r[0]), ry2 = make_float2(r[1], r[1]);
  const float2 a0 = make_float2(m[0], m[4]), a1 = make_float2(m[1], m[5]);
  const float2 b0 = make_float2(m[2], m[6]), b1 = make_float2(m[3], m[7]);
  const float2 dxa = sub2(a1, a0), dxb = sub2(b1, b0);
  const float2 ca = fma2(rx2, dxa, a0), cb = fma2(rx2, dxb, b0);
  const float2 dy = sub2(cb, ca);
  const float2 c = fma2(ry2, dy, ca);
  const float dz = c.y - c.x;
  if (GRAD) {
    gz = dz;
    gy = fmaf(rz, dy.y - dy.x, dy.x);
    const float2 e = fma2(ry2, sub2(dxb, dxa), dxa);
    gx = fmaf(rz, e.y - e.x, e.x);
  }
  return fmaf(rz, dz, c.x);
}

// ------------------------------------------------------- Parzen window
// Cubic B-spline weights of the four bins floor(c)-1 .. floor(c)+2 for
// fraction t = c - floor(c), each multiplied by `scale`.
__device__ __forceinline__ void bspline4(float t, float scale, float w[4]) {
  const float u = 1.0f - t;
  const float t2 = t * t, u2 = u * u;
  const float t3 = t2 * t, u3 = u2 * u;
  const float s6 = scale * (1.0f / 6.0f), s23 = scale * (2.0f / 3.0f), sh = 0.5f * scale;
  w[0] = u3 * s6;
  w[1] = fmaf(t3, sh, fmaf(-t2, scale, s23));
  w[2] = fmaf(u3, sh, fmaf(-u2, scale, s23));
  w[3] = t3 * s6;
}

// d beta(s)/ds at s = bin - c for the same four bins.
__device__ __forceinline__ void bspline4_deriv(float t, float d[4]) {
  const float u = 1.0f - t;
  d[0] = 0.5f * u * u;
  d[1] = t * fmaf(-1.5f, t, 2.0f);
  d[2] = u * fmaf(1.5f, u, -2.0f);
  d[3] = -0.5f * t * t;
}

// Bin coordinate c = 2 + (clamp(v, lo, hi) - lo) * sc, sc = (B-5)/(hi-lo).
// Subtracting lo first keeps c inside [2, B-3] up to one rounding of
// (hi-lo)*sc, whatever the magnitude of lo, so every histogram / table
// address derived from floor(c) stays in range (NaN clamps to lo).
struct BinMap {
  float lo, hi, sc, off;
};

__device__ __forceinline__ float bin_coord(const BinMap& m, float v) {
  return fmaf(fminf(fmaxf(v, m.lo), m.hi) - m.lo, m.sc, 2.0f);
}

// --------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One fixed-image value as float.
__device__ __forceinline__ float load1(const float* __restrict__ p) { return __ldg(p); }
__device__ __forceinline__ float load1(const __half* __restrict__ p) { return __half2float(__ldg(p)); }

}  // namespace ffdp
