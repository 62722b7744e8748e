// k_lncc.cu -- LNCC forward + backward for windows up to 7 on a materialised
// warped image J: writes g = dL/dJ per voxel (stand-alone LNCC) or, in the
// objective, adds the MI partial gradient and runs the sampler backward (du
// and the affine partials) from the stored slope.
// Wider windows run as separable passes (k_lncc_wide.cu).
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
// Work layout.  A CTA owns a 32 x TY column of output voxels and streams a z
// segment of planes; each thread keeps the values of its staged positions of
// the halo plane for the last w planes in registers, so the z window sums
// need no shared memory and shared memory carries only the x and y passes.
// The five window sums run on packed fp32 pairs ((S_J, S_F), (S_JJ, S_FF))
// plus S_FJ.  CTAs are persistent over tiles, so the per-CTA partial records
// stay O(#SMs).  Two forms:
//   * split (the default): k_lncc_fw computes the window sums, cc and the
//     three g-terms at the tile's own outputs (an R halo) and stores the
//     g-terms; k_lncc_bw sums them over the window (an R halo again) and runs
//     the epilogue.  Each kernel holds about half the state of the fused one
//     (80 registers, three CTAs per SM) and has two barriers per plane.
//   * fused (FFDP_LNCC_FUSED, and the halo-recompute build): k_lncc_rh does
//     both halves per plane on a 2R halo, the g-terms never leaving the chip.
#include <type_traits>

#include "ffdp_internal.h"
#include "ffdp_lncc.cuh"

namespace ffdp {

constexpr int kTX = kLnccTX;

template <int R>
struct LT {
  static constexpr int W = 2 * R + 1;
  static constexpr int TY = lncc_ty(R);
  static constexpr int E2W = kTX + 4 * R;  // multiple of 4
  static constexpr int E2H = TY + 4 * R;
  static constexpr int E1W = kTX + 2 * R;
  static constexpr int E1H = TY + 2 * R;
  static constexpr int E1S = (E1W + 3) & ~3;
  static constexpr int XB = E2H * E1S * 5;
  static constexpr int PAD = 32;
  static_assert(E1H * kTX * 3 <= XB, "g-term x buffer must fit in the x buffer");
  static_assert((TY % 4) == 0, "TY multiple of 4");
};

template <int R>
struct LTR;

// LN_DU: the stored slope dJ/dq of a later step's output plane (TY x 32
// voxels, 3 floats each), staged in shared memory by asynchronous copies so
// that the epilogue does not wait on DRAM.  Three slots: the copy for step
// s + 1 is issued at the start of step s, waited for (by its issuing thread)
// before the first barrier of step s + 1 and read after it; its slot was
// last read in step s - 2, before the first barrier of step s - 1.
template <int TY>
struct SlopeStage {
  static constexpr int ROW = 3 * kTX;       // floats per staged row
  static constexpr int SLOT = TY * ROW;     // floats per slot
  static constexpr int FLOATS = 3 * SLOT;   // three slots
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

// Issue the copies of one output plane (none if src is null) of the tile into
// slot, then commit one group (possibly empty).  src: the slope of the tile's
// first voxel in that plane; rs: floats per grid row.  Full tiles of a grid
// whose rows are a multiple of 4 voxels (every tile row then starts 16-byte
// aligned) take 16-byte copies, 24 per row; edge tiles and other widths take
// 4-byte copies.
template <int TY, int NT>
__device__ __forceinline__ void stage_slope(float* slot, const float* src, const Geom& g, int x0, int y0, bool full,
                                            int tid) {
  constexpr int ROW = SlopeStage<TY>::ROW;
  const size_t rs = 3 * (size_t)g.fW;
  if (src) {
    if (full) {
      constexpr int CPR = ROW / 4;
#pragma unroll
      for (int c0 = 0; c0 < TY * CPR; c0 += NT) {
        const int c = c0 + tid;
        if (c < TY * CPR) {
          const int r = c / CPR, k = c - r * CPR;
          cp_async16(slot + r * ROW + 4 * k, src + r * rs + 4 * k);
        }
      }
    } else {
      const int ncol = min(kTX, g.fW - x0), nrow = min(TY, g.fH - y0);
      const int cpr = 3 * ncol;
      for (int c = tid; c < nrow * cpr; c += NT) {
        const int r = c / cpr, k = c - r * cpr;
        cp_async4(slot + r * ROW + k, src + r * rs + k);
      }
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Streamed (J, F) reads of the staged halo positions: read once per CTA, so
// they bypass L1 (no allocation) and leave it to the MI table cells.
__device__ __forceinline__ float ld_stream(const float* p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_stream(const __half* p) {
  unsigned short v;
  asm("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(v) : "l"(p));
  return __half2float(__ushort_as_half(v));
}

// all but the most recent group of this thread's copies have landed
__device__ __forceinline__ void slope_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <int R, bool DU>
static size_t smem_of();

// Work of one CTA: an equal share (a.per planes) of the sequence of (column,
// plane) pairs, columns outermost, cut at column boundaries into z segments.
// Every segment costs 4R extra planes of window halo, against a round-robin
// of fixed z chunks whose last round leaves most CTAs idle.
struct LnccSegs {
  long long u, end;
  int D, tilesX;
  __device__ explicit LnccSegs(const LnccArgs& a) : D(a.g.fD), tilesX(a.tilesX) {
    const long long total = (long long)a.tilesX * a.tilesY * a.g.fD;
    u = (long long)blockIdx.x * a.per;
    end = min(total, u + a.per);
  }
  __device__ bool next(int& tx, int& ty, int& z0, int& z1) {
    if (u >= end) return false;
    const long long col = u / D;
    z0 = (int)(u - col * D);
    z1 = (int)min((long long)D, z0 + (end - u));
    tx = (int)(col % tilesX);
    ty = (int)(col / tilesX);
    u += z1 - z0;
    return true;
  }
};

// Plane-synchronous work order: in full rounds every CTA takes one whole tile
// column (all planes), so neighbouring tiles pass the same planes at about the
// same time and read each other's halo rows from L2; the columns left over
// after the last full round are shared as equal runs of (column, plane) pairs.
struct LnccSegsSync {
  long long u, end;
  int D, tilesX, G, b, r, rounds;
  __device__ explicit LnccSegsSync(const LnccArgs& a) : D(a.g.fD), tilesX(a.tilesX) {
    const int ncols = a.tilesX * a.tilesY;
    G = gridDim.x;
    b = blockIdx.x;
    rounds = ncols / G;
    r = 0;
    const long long rem = (long long)(ncols - rounds * G) * D;
    const long long per = (rem + G - 1) / G;
    const long long base = (long long)rounds * G * D;
    u = base + (long long)b * per;
    end = min(base + rem, u + per);
  }
  __device__ bool next(int& tx, int& ty, int& z0, int& z1) {
    if (r < rounds) {
      const int col = r * G + b;
      ++r;
      tx = col % tilesX;
      ty = col / tilesX;
      z0 = 0;
      z1 = D;
      return true;
    }
    if (u >= end) return false;
    const long long col = u / D;
    z0 = (int)(u - col * D);
    z1 = (int)min((long long)D, z0 + (end - u));
    tx = (int)(col % tilesX);
    ty = (int)(col / tilesX);
    u += z1 - z0;
    return true;
  }
};
// The split forward kernel takes the plane-synchronous order (its halo reads
// then come from L2: 1.14 -> 1.12 ms at 512^3); the backward kernel keeps the
// equal runs (plane-synchronous, its sampler-backward epilogue slowed from
// 1.72 to 2.35 ms, as in the fused kernel).
using SegsFw = LnccSegsSync;
using SegsBw = LnccSegs;

// Sampler backward in the window kernel's epilogue (LN_DU), from the slope
// dJ/dq that the sampling sweep stored: per voxel e = g dJ/dq with g = dL/dJ,
// du = K^T e, and the affine moments sum e_r and sum e_r (i_c - ctr_c).  A
// thread's outputs keep their column and rows over a z segment, so its x and
// y moments follow from per-row sums at fold time; only the z moment is
// accumulated per voxel.  Folded into the CTA's fp64 records every 32 planes
// and at the end of each segment.
template <int NOUT>
struct DuAcc {
  float S[NOUT][3];  // sum of e_r per output row
  float Zm[3];       // sum of e_r (iz - ctr_z)
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int r = 0; r < 3; ++r) {
#pragma unroll
      for (int k = 0; k < NOUT; ++k) S[k][r] = 0.0f;
      Zm[r] = 0.0f;
    }
  }
  // q: the voxel's staged slope (shared memory)
  __device__ __forceinline__ void add(const LnccArgs& a, int k, size_t lin, const float* q, float cz, float gv) {
    const float e0 = gv * q[0], e1 = gv * q[1], e2 = gv * q[2];
    if (a.du) {
      const float* K = a.g.K;
      float* d = a.du + 3 * lin;
      if (a.g.k_diag) {
        d[0] = K[0] * e0;
        d[1] = K[4] * e1;
        d[2] = K[8] * e2;
      } else {
        d[0] = fmaf(K[0], e0, fmaf(K[3], e1, K[6] * e2));
        d[1] = fmaf(K[1], e0, fmaf(K[4], e1, K[7] * e2));
        d[2] = fmaf(K[2], e0, fmaf(K[5], e1, K[8] * e2));
      }
    }
    S[k][0] += e0;
    S[k][1] += e1;
    S[k][2] += e2;
    Zm[0] = fmaf(e0, cz, Zm[0]);
    Zm[1] = fmaf(e1, cz, Zm[1]);
    Zm[2] = fmaf(e2, cz, Zm[2]);
  }
  // warp-uniform; ws = this warp's fp64 record, cx / cy = centred column / rows
  __device__ __forceinline__ void fold(double* ws, int lane, float cx, const float cy[NOUT]) {
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      float s = S[0][r], ym = S[0][r] * cy[0];
#pragma unroll
      for (int k = 1; k < NOUT; ++k) {
        s += S[k][r];
        ym = fmaf(S[k][r], cy[k], ym);
      }
      const float v0 = warp_sum(s), v1 = warp_sum(s * cx), v2 = warp_sum(ym), v3 = warp_sum(Zm[r]);
      if (lane == 0) {
        ws[kPS + r] += (double)v0;
        ws[kPM + 3 * r] += (double)v1;
        ws[kPM + 3 * r + 1] += (double)v2;
        ws[kPM + 3 * r + 2] += (double)v3;
      }
#pragma unroll
      for (int k = 0; k < NOUT; ++k) S[k][r] = 0.0f;
      Zm[r] = 0.0f;
    }
  }
};

// ------------------------------------------------- register-history variant
// Same mathematics and tiling, for R <= 3.  Each thread stages NSTG fixed
// positions of the 2R-halo plane (its own NOUT output voxels first) and keeps
// their (J, F) for the last w planes in registers, so the z window sums need
// no shared memory; the z sums of the g-terms run over a register ring of the
// thread's own outputs.  Shared memory carries only the x and y passes:
//   [B] z sums (registers) -> zbuf,        [C] x sums zbuf -> xbuf,
//   [D] y sums, cc and g-terms -> gbuf,    [E] x sums gbuf -> gxbuf,
//   [F] y sums at the thread's outputs -> register ring, [G] z sums, dJ.
// The plane loop is unrolled by w so that every register slot index is a
// compile-time constant.
template <int R>
struct LTR {
  using L = LT<R>;
  static constexpr int W = L::W, TY = L::TY, E2W = L::E2W, E2H = L::E2H;
  static constexpr int NOUT = TY * kTX / kLnccRHThreads;       // outputs per thread
  static constexpr int NCORE = TY * kTX;
  static constexpr int NHALO = E2H * E2W - NCORE;        // halo positions outside the outputs
  static constexpr int NEXTRA = (NHALO + kLnccRHThreads - 1) / kLnccRHThreads;
  static constexpr int NSTG = NOUT + NEXTRA;
  static_assert(NOUT * kLnccRHThreads == NCORE, "outputs per thread");
  // Row stride of the z-sum buffer: the x pass reads 2-output items (16 bytes
  // of (S_J, S_F) pairs, 8 bytes of S_FJ per lane), E1S/2 items per row; the
  // stride makes a row continue the bank sequence of the previous one, so
  // lanes that cross a row boundary inside a warp do not collide.
  static constexpr int XG = L::E1S / 2;
  static constexpr int zs_of(int s) { return (s % 2 == 0 && ((s / 2 - XG) % 16 + 16) % 16 == 0) ? s : zs_of(s + 1); }
  static constexpr int ZS = zs_of(L::E2W);
  static constexpr int ZB = L::E2H * ZS * 5;
  // shared memory: zbuf (z sums, later the g-terms) and xbuf (x sums, later
  // the x-summed g-terms); no plane ring
  static constexpr int OFF_Z = 0;
  static constexpr int OFF_X = ZB + L::PAD;
  static constexpr int TOTAL = OFF_X + L::XB + L::PAD;
  static_assert(L::E1H * L::E1S * 3 <= ZB, "g-term plane must fit in the z buffer");
  static_assert(OFF_X % 4 == 0, "16-byte alignment");
};

// Halo position h (outside the output core) of a tile: the top and bottom 2R
// rows in full, then the 2R columns on either side of the core rows.
template <int R>
__device__ __forceinline__ void halo_pos(int h, int& row, int& col) {
  using L = LT<R>;
  constexpr int STRIP = 2 * R * L::E2W;
  if (h < STRIP) {
    row = h / L::E2W;
    col = h - row * L::E2W;
  } else if (h < 2 * STRIP) {
    h -= STRIP;
    row = 2 * R + L::TY + h / L::E2W;
    col = h % L::E2W;
  } else {
    h -= 2 * STRIP;
    row = 2 * R + h / (4 * R);
    const int c = h % (4 * R);
    col = c < 2 * R ? c : kTX + c;
  }
}

template <typename FT, int BMAX, int R, bool DU>
__global__ void __launch_bounds__(kLnccRHThreads, FFDP_LNCC_MINB) k_lncc_rh(const LnccArgs a) {
  using L = LT<R>;
  using Q = LTR<R>;
  constexpr int W = L::W, TY = L::TY, E2S = Q::ZS;
  constexpr int E1W = L::E1W, E1H = L::E1H, E1S = L::E1S;
  constexpr int NOUT = Q::NOUT, NSTG = Q::NSTG;
  constexpr bool MI = BMAX != 0;

  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ double wsum[kLnccRHThreads / 32][13];
  float2* zP = reinterpret_cast<float2*>(sm + Q::OFF_Z);
  float2* zQ = zP + L::E2H * E2S;
  float* zX = sm + Q::OFF_Z + 4 * L::E2H * E2S;
  float2* xP = reinterpret_cast<float2*>(sm + Q::OFF_X);
  float2* xQ = xP + L::E2H * E1S;
  float* xX = sm + Q::OFF_X + 4 * L::E2H * E1S;
  float2* gP = reinterpret_cast<float2*>(sm + Q::OFF_Z);
  float* gX = sm + Q::OFF_Z + 2 * E1H * E1S;
  float2* gxP = reinterpret_cast<float2*>(sm + Q::OFF_X);
  float* gxX = sm + Q::OFF_X + 2 * E1H * kTX;
  float* slope = sm + Q::TOTAL;  // LN_DU only

  const Geom& g = a.g;
  const int tid = threadIdx.x;
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const float inv_n = a.inv_n, eps = a.eps, gs = a.gscale;
  const float2 ninv2 = make_float2(-inv_n, -inv_n);
  const size_t plane = (size_t)g.fW * g.fH;
  float cc_acc = 0.0f;
  if ((tid & 31) == 0)
    for (int q = 0; q < 13; ++q) wsum[tid >> 5][q] = 0.0;
  DuAcc<NOUT> dacc;
  dacc.clear();

  // staged positions: shared-memory index in the halo plane and in-plane
  // global offset (-1: outside the grid, read as zero; -2: no position)
  const int ox = tid & 31, oy0 = (tid >> 5) * NOUT;
  int sidx[NSTG];
#pragma unroll
  for (int i = 0; i < NSTG; ++i) {
    int row, col;
    if (i < NOUT) {
      row = oy0 + i + 2 * R;
      col = ox + 2 * R;
    } else {
      const int h = tid + (i - NOUT) * kLnccRHThreads;
      if (h < Q::NHALO) {
        halo_pos<R>(h, row, col);
      } else {
        row = -1;
        col = 0;
      }
    }
    sidx[i] = row < 0 ? -1 : row * E2S + col;
  }

  float2 hist[W][NSTG];  // (J, F) of the last w planes at the staged positions
  float2 grP[W][NOUT];   // g-term 2-D window sums at the own outputs, last w planes
  float grX[W][NOUT];
  float2 nxt[NSTG];      // next plane, fetched one step ahead
  int soff[NSTG];
  constexpr bool RC = DU && kLnccRecompute;  // J and its slope sampled here, nothing stored
  const FT* __restrict__ Mp = static_cast<const FT*>(a.M);
  // J at fixed-grid voxel (x, y, z) (and its slope dJ/dq when GRAD), sampled
  // from M and u like the sweeps do
  auto sample = [&](int x, int y, int z, size_t lin, float* dq, auto grad) -> float {
    constexpr bool GRAD = decltype(grad)::value;
    float u0 = 0.0f, u1 = 0.0f, u2 = 0.0f;
    if (a.u) {
      u0 = __ldg(a.u + 3 * lin);
      u1 = __ldg(a.u + 3 * lin + 1);
      u2 = __ldg(a.u + 3 * lin + 2);
    }
    int b[3];
    float r[3], m[8];
    if (g.ia) {
      cell_of_int(g, x, y, z, u0, u1, u2, b, r);
    } else {
      long long P[3];
      anchor(g, x, y, z, P);
      cell_of(g, P, u0, u1, u2, b, r);
    }
    gather8<FT>(Mp, g, b, m);
#pragma unroll
    for (int q = 0; q < 8; ++q) m[q] = tap_value<FT>(m[q]);
    float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f;
    const float jv = interp8<GRAD>(m, r, d0, d1, d2);
    if (GRAD) {
      dq[0] = d0;
      dq[1] = d1;
      dq[2] = d2;
    }
    return jv;
  };

  auto load_plane = [&](int zp) {
    const bool zin = zp >= 0 && zp < g.fD;
    const size_t base = (size_t)zp * plane;
#pragma unroll
    for (int i = 0; i < NSTG; ++i) {
      float2 v = make_float2(0.0f, 0.0f);
      if (zin && soff[i] >= 0) {
        if constexpr (RC) {
          const int y = (int)fast_div((unsigned)soff[i], g.divW_m, g.divW_s);
          v.x = sample(soff[i] - y * g.fW, y, zp, base + soff[i], nullptr, std::false_type{});
        } else {
          v.x = ld_stream(a.J + base + soff[i]);
        }
        v.y = ld_stream(F + base + soff[i]);
      }
      nxt[i] = v;
    }
  };

  LnccSegs seg(a);
  int tx, ty, z0, z1;
  while (seg.next(tx, ty, z0, z1)) {
    const int x0 = tx * kTX, y0 = ty * TY;
    const int nsteps = (z1 - z0) + 4 * R;
    // LN_DU: the tile's slope (plane stride slope_plane) and its staging slots;
    // slot_rd is the slot of the current step's output plane (s mod 3)
    const bool full = x0 + kTX <= g.fW && y0 + TY <= g.fH && (g.fW & 3) == 0;
    const size_t slope_plane = 3 * (size_t)g.fW * g.fH;
    const float* slope_tile = DU ? a.dJdq + 3 * ((size_t)y0 * g.fW + x0) : nullptr;
    int slot_rd = 2;
    auto fold_du = [&] {
      float cy[NOUT];
#pragma unroll
      for (int k = 0; k < NOUT; ++k) cy[k] = (float)(y0 + oy0 + k) - g.ctr[1];
      dacc.fold(wsum[tid >> 5], tid & 31, (float)(x0 + ox) - g.ctr[0], cy);
    };
#pragma unroll
    for (int i = 0; i < NSTG; ++i) {
      soff[i] = -2;
      if (sidx[i] >= 0) {
        const int row = sidx[i] / E2S, col = sidx[i] - row * E2S;
        const int x = x0 - 2 * R + col, y = y0 - 2 * R + row;
        soff[i] = ((unsigned)x < (unsigned)g.fW && (unsigned)y < (unsigned)g.fH) ? y * g.fW + x : -1;
      }
    }
#pragma unroll
    for (int q = 0; q < W; ++q) {
#pragma unroll
      for (int k = 0; k < NOUT; ++k) {
        grP[q][k] = make_float2(0.f, 0.f);
        grX[q][k] = 0.f;
      }
    }
    load_plane(z0 - 2 * R);

    for (int s0 = 0; s0 < nsteps; s0 += W) {
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int s = s0 + j;
        if (s < nsteps) {
          const int zi = z0 - 2 * R + s;
          const bool pass1 = s >= 2 * R;
          const bool pass2 = s >= 4 * R;
          // the fetched plane becomes the newest history slot j; fetch the next
#pragma unroll
          for (int i = 0; i < NSTG; ++i) hist[j][i] = nxt[i];
          if (s + 1 < nsteps) load_plane(zi + 1);
          if constexpr (DU && !RC) {
            slot_rd = slot_rd == 2 ? 0 : slot_rd + 1;
            const int sn = s + 1;  // the output plane of the next step
            const float* src =
                (sn >= 4 * R && sn < nsteps) ? slope_tile + (size_t)(zi + 1 - 2 * R) * slope_plane : nullptr;
            stage_slope<TY, kLnccRHThreads>(slope + (slot_rd == 2 ? 0 : slot_rd + 1) * SlopeStage<TY>::SLOT, src,
                                            g, x0, y0, full, tid);
          }
          if (pass1) {
            // [B] z sums over the register history -> zbuf
#pragma unroll
            for (int i = 0; i < NSTG; ++i) {
              if (sidx[i] >= 0) {
                float2 sP = hist[0][i];
                float2 sQ = mul2(hist[0][i], hist[0][i]);
                float sX = hist[0][i].x * hist[0][i].y;
#pragma unroll
                for (int q = 1; q < W; ++q) {
                  sP = add2(sP, hist[q][i]);
                  sQ = fma2(hist[q][i], hist[q][i], sQ);
                  sX = fmaf(hist[q][i].x, hist[q][i].y, sX);
                }
                zP[sidx[i]] = sP;
                zQ[sidx[i]] = sQ;
                zX[sidx[i]] = sX;
              }
            }
          }
          if constexpr (DU && !RC) slope_wait_prev();
          __syncthreads();
          if (pass1) {
            // [C] x sums, 2 outputs per item: neighbouring lanes read
            // neighbouring 16-byte vectors (no bank conflicts)
            constexpr int XG = E1S / 2;
            constexpr int NI = 2 + 2 * R;  // inputs of a 2-output run
            for (int it = tid; it < L::E2H * XG; it += kLnccRHThreads) {
              const int row = it / XG, g2 = it - row * XG;
              float2 vP[NI], vQ[NI];
              float vX[NI];
              const float4* sP4 = reinterpret_cast<const float4*>(zP + row * E2S + 2 * g2);
              const float4* sQ4 = reinterpret_cast<const float4*>(zQ + row * E2S + 2 * g2);
              const float2* sX2 = reinterpret_cast<const float2*>(zX + row * E2S + 2 * g2);
#pragma unroll
              for (int k = 0; k < NI / 2; ++k) {
                const float4 p = sP4[k], q = sQ4[k];
                const float2 x = sX2[k];
                vP[2 * k] = make_float2(p.x, p.y);
                vP[2 * k + 1] = make_float2(p.z, p.w);
                vQ[2 * k] = make_float2(q.x, q.y);
                vQ[2 * k + 1] = make_float2(q.z, q.w);
                vX[2 * k] = x.x;
                vX[2 * k + 1] = x.y;
              }
              float2 aP = vP[0], aQ = vQ[0];
              float aX = vX[0];
#pragma unroll
              for (int k = 1; k <= 2 * R; ++k) {
                aP = add2(aP, vP[k]);
                aQ = add2(aQ, vQ[k]);
                aX += vX[k];
              }
              const float2 bP = sub2(add2(aP, vP[2 * R + 1]), vP[0]);
              const float2 bQ = sub2(add2(aQ, vQ[2 * R + 1]), vQ[0]);
              const float bX = (aX + vX[2 * R + 1]) - vX[0];
              *reinterpret_cast<float4*>(xP + row * E1S + 2 * g2) = make_float4(aP.x, aP.y, bP.x, bP.y);
              *reinterpret_cast<float4*>(xQ + row * E1S + 2 * g2) = make_float4(aQ.x, aQ.y, bQ.x, bQ.y);
              *reinterpret_cast<float2*>(xX + row * E1S + 2 * g2) = make_float2(aX, bX);
            }
          }
          __syncthreads();
          if (pass1) {
            // [D] y sums -> window sums at plane zc on the R-halo region; cc and
            // g-terms.  Runs of 3 rows per item (one round of items for the
            // CTA); rows are read as the window slides, keeping only the two
            // rows that leave it.
            constexpr int RUN = 3;
            constexpr int YR = (E1H + RUN - 1) / RUN;
            const int zc = zi - R;
            const bool zin = zc >= 0 && zc < g.fD;
            const bool zown = zc >= z0 && zc < z1;
            for (int it = tid; it < E1W * YR; it += kLnccRHThreads) {
              const int x1 = it % E1W, ys = RUN * (it / E1W);
              auto rowP = [&](int row) { return row < L::E2H ? xP[row * E1S + x1] : make_float2(0.f, 0.f); };
              auto rowQ = [&](int row) { return row < L::E2H ? xQ[row * E1S + x1] : make_float2(0.f, 0.f); };
              auto rowX = [&](int row) { return row < L::E2H ? xX[row * E1S + x1] : 0.f; };
              float2 oP[RUN - 1], oQ[RUN - 1];
              float oX[RUN - 1];
#pragma unroll
              for (int k = 0; k < RUN - 1; ++k) {
                oP[k] = rowP(ys + k);
                oQ[k] = rowQ(ys + k);
                oX[k] = rowX(ys + k);
              }
              float2 aP = oP[0], aQ = oQ[0];
              float aX = oX[0];
#pragma unroll
              for (int k = 1; k <= 2 * R; ++k) {
                const float2 p = k < RUN - 1 ? oP[k] : rowP(ys + k);
                const float2 q = k < RUN - 1 ? oQ[k] : rowQ(ys + k);
                const float x = k < RUN - 1 ? oX[k] : rowX(ys + k);
                aP = add2(aP, p);
                aQ = add2(aQ, q);
                aX += x;
              }
              const int x = x0 - R + x1;
              const bool xin = (unsigned)x < (unsigned)g.fW;
              const bool xown = x1 >= R && x1 < R + kTX;
#pragma unroll
              for (int k = 0; k < RUN; ++k) {
                if (k > 0) {
                  aP = sub2(add2(aP, rowP(ys + 2 * R + k)), oP[k - 1]);
                  aQ = sub2(add2(aQ, rowQ(ys + 2 * R + k)), oQ[k - 1]);
                  aX = (aX + rowX(ys + 2 * R + k)) - oX[k - 1];
                }
                const int y1 = ys + k;
                if (y1 < E1H) {
                  const int y = y0 - R + y1;
                  float2 gpair = make_float2(0.f, 0.f);
                  float gfj = 0.f;
                  if (zin && xin && (unsigned)y < (unsigned)g.fH) {
                    // aP = (S_J, S_F), aQ = (S_JJ, S_FF), aX = S_FJ; variances clamped at 0
                    float2 v = fma2(mul2(aP, aP), ninv2, aQ);
                    v = make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f));
                    const float cross = fmaf(-aP.x * aP.y, inv_n, aX);
                    const float D = fmaf(v.x, v.y, eps);
                    const float rD = rcp_approx(D);
                    const float A1 = 2.0f * cross * rD;
                    const float cc = cross * cross * rD;
                    const float A2 = cc * v.y * rD;
                    gfj = gs * A1;
                    gpair.y = -gs * A2;
                    gpair.x = gs * (2.0f * A2 * aP.x - A1 * aP.y) * inv_n;
                    if (zown && xown && y1 >= R && y1 < R + TY) cc_acc += cc;
                  }
                  gP[y1 * E1S + x1] = gpair;
                  gX[y1 * E1S + x1] = gfj;
                }
              }
            }
          }
          __syncthreads();
          if (pass1) {
            // [E] x sums of the g-terms onto the 32 output columns, 2 per item
            constexpr int XG2 = kTX / 2;
            constexpr int NI = 2 + 2 * R;
            for (int it = tid; it < E1H * XG2; it += kLnccRHThreads) {
              const int row = it / XG2, g2 = it - row * XG2;
              float2 vP[NI];
              float vX[NI];
              const float4* sP4 = reinterpret_cast<const float4*>(gP + row * E1S + 2 * g2);
              const float2* sX2 = reinterpret_cast<const float2*>(gX + row * E1S + 2 * g2);
#pragma unroll
              for (int k = 0; k < NI / 2; ++k) {
                const float4 p = sP4[k];
                const float2 x = sX2[k];
                vP[2 * k] = make_float2(p.x, p.y);
                vP[2 * k + 1] = make_float2(p.z, p.w);
                vX[2 * k] = x.x;
                vX[2 * k + 1] = x.y;
              }
              float2 aP = vP[0];
              float aX = vX[0];
#pragma unroll
              for (int k = 1; k <= 2 * R; ++k) {
                aP = add2(aP, vP[k]);
                aX += vX[k];
              }
              const float2 bP = sub2(add2(aP, vP[2 * R + 1]), vP[0]);
              const float bX = (aX + vX[2 * R + 1]) - vX[0];
              *reinterpret_cast<float4*>(gxP + row * kTX + 2 * g2) = make_float4(aP.x, aP.y, bP.x, bP.y);
              *reinterpret_cast<float2*>(gxX + row * kTX + 2 * g2) = make_float2(aX, bX);
            }
          }
          __syncthreads();
          // [F] y sums of the g-terms at the own outputs -> register ring slot j
          if (pass1) {
            float2 vP[NOUT + 2 * R];
            float vX[NOUT + 2 * R];
#pragma unroll
            for (int k = 0; k < NOUT + 2 * R; ++k) {
              vP[k] = gxP[(oy0 + k) * kTX + ox];
              vX[k] = gxX[(oy0 + k) * kTX + ox];
            }
            float2 aP = vP[0];
            float aX = vX[0];
#pragma unroll
            for (int k = 1; k <= 2 * R; ++k) {
              aP = add2(aP, vP[k]);
              aX += vX[k];
            }
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              if (k > 0) {
                aP = sub2(add2(aP, vP[2 * R + k]), vP[k - 1]);
                aX = (aX + vX[2 * R + k]) - vX[k - 1];
              }
              grP[j][k] = aP;
              grX[j][k] = aX;
            }
          } else {
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              grP[j][k] = make_float2(0.f, 0.f);
              grX[j][k] = 0.f;
            }
          }
          // [G] z sums over the register ring -> dJ at plane zo = zi - 2R
          if (pass2) {
            const int zo = zi - 2 * R;
            const int OLD = (j + 1) % W;  // history slot of plane zo
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              float2 bP = grP[0][k];
              float bX = grX[0][k];
#pragma unroll
              for (int q = 1; q < W; ++q) {
                bP = add2(bP, grP[q][k]);
                bX += grX[q][k];
              }
              const float jv = hist[OLD][k].x, fv = hist[OLD][k].y;
              const int X = x0 + ox, Y = y0 + oy0 + k;
              if (X < g.fW && Y < g.fH) {
                float gv = fmaf(fv, bX, fmaf(2.0f * jv, bP.y, bP.x));
                if (MI) gv += mi_grad_ln<(MI ? BMAX : 32)>(a.T, a.bf, a.bj, fv, jv);
                const size_t lin = ((size_t)zo * g.fH + Y) * g.fW + X;
                if constexpr (RC) {
                  float q[3];
                  sample(X, Y, zo, lin, q, std::true_type{});
                  dacc.add(a, k, lin, q, (float)zo - g.ctr[2], gv);
                } else if constexpr (DU)
                  dacc.add(a, k, lin, slope + slot_rd * SlopeStage<TY>::SLOT + (oy0 + k) * SlopeStage<TY>::ROW + 3 * ox,
                           (float)zo - g.ctr[2], gv);
                else if (a.dJ)
                  a.dJ[lin] = gv;
              }
            }
          }
          // fold the fp32 cc (and affine) partials into fp64 every 32 planes
          // (uniform across the CTA)
          if ((s & 31) == 31) {
            const float v = warp_sum(cc_acc);
            if ((tid & 31) == 0) wsum[tid >> 5][12] += (double)v;
            cc_acc = 0.0f;
            if constexpr (DU) fold_du();
          }
        }
      }
    }
    if constexpr (DU) fold_du();  // the next segment has other columns and rows
  }
  {
    const float v = warp_sum(cc_acc);
    if ((tid & 31) == 0) wsum[tid >> 5][12] += (double)v;
  }
  __syncthreads();
  if (tid < kPartialStride) {
    double s = 0.0;
    if (tid == kPCC || (DU && tid < 12))
      for (int k = 0; k < kLnccRHThreads / 32; ++k) s += wsum[k][tid];
    a.partials[(size_t)blockIdx.x * kPartialStride + tid] = s;
  }
}

// ---------------------------------------------------------- split variant
// The same mathematics in two kernels, so that each holds half the state:
//   forward (k_lncc_fw): the five window sums at the tile's own outputs only
//     (an R halo instead of 2R), cc and the three g-terms, stored per voxel
//     ([3][N], 12 B/voxel of workspace);
//   backward (k_lncc_bw): the window sums of the stored g-terms at the tile's
//     outputs (again an R halo), dL/dJ with the MI term, then dL/dJ stored or
//     the sampler backward from the stored slope.
// Each has two barriers per plane, and in both the thread that owns an output
// does its y sums itself (no work items in that pass).
template <int R>
struct LTS {
  static constexpr int W = 2 * R + 1;
  static constexpr int TY = lncc_ty(R);
  static constexpr int HW = kTX + 2 * R;  // R-halo plane: HH rows of HW columns
  static constexpr int HH = TY + 2 * R;
  static constexpr int NOUT = TY * kTX / kLnccRHThreads;
  static constexpr int NCORE = TY * kTX;
  static constexpr int NHALO = HH * HW - NCORE;
  static constexpr int NEXTRA = (NHALO + kLnccRHThreads - 1) / kLnccRHThreads;
  static constexpr int NSTG = NOUT + NEXTRA;
  static_assert(NOUT * kLnccRHThreads == NCORE, "outputs per thread");
  // The forward x pass takes items of four outputs, one per thread in a
  // single round (rows padded to RB, a multiple of 8, per column group),
  // consecutive threads on consecutive rows; the backward one, whose thread
  // state leaves no room for eight pairs at once, items of two outputs
  // (consecutive threads along a row, two rounds).  The row strides are odd
  // multiples of 16 bytes (halo plane: 66 pairs; x sums: 34 pairs, 36
  // scalars), so that the eight lanes of every 16-byte access phase fall on
  // distinct banks in both.
  static constexpr int ZS = 66, XS = 34, XSX = 36;
  static_assert(HW <= ZS, "halo row fits the row stride");
  static constexpr int XG4 = kTX / 4;
  static constexpr int RB = (HH + 7) / 8 * 8;
  static_assert(RB * XG4 <= kLnccRHThreads, "x items: one round");
  // forward: z sums (5 channels) on the halo plane, x sums (5) on HH x 32
  static constexpr int FW_Z = HH * ZS * 5;
  static constexpr int FW_TOTAL = FW_Z + HH * (4 * XS + XSX);
  // backward: g-terms (3 channels) on the halo plane, x sums (3) on HH x 32
  static constexpr int BW_G = HH * ZS * 3;
  static constexpr int BW_TOTAL = BW_G + HH * (2 * XS + XSX);
  static_assert(FW_Z % 4 == 0 && BW_G % 4 == 0 && BW_TOTAL % 4 == 0, "16-byte aligned regions");
};

// Box sums of width 2R + 1 at four consecutive outputs from v[0 .. 2R + 3],
// as sums of shared partial sums (no running add-and-subtract: the moments'
// variances cancel, and every subtraction of a sliding window would add its
// rounding error to them).
__device__ __forceinline__ float addv(float a, float b) { return a + b; }
__device__ __forceinline__ float2 addv(float2 a, float2 b) { return add2(a, b); }
template <int R, typename T>
__device__ __forceinline__ void win4(const T* v, T o[4]) {
  const T a = addv(v[1], v[2]);                 // in windows 0, 1
  const T b = addv(v[2 * R + 1], v[2 * R + 2]);  // in windows 2, 3
  o[0] = addv(v[0], a);
  o[1] = addv(a, v[2 * R + 1]);
  o[2] = addv(v[2], b);
  o[3] = addv(b, v[2 * R + 3]);
  if constexpr (R >= 2) {
    T c = v[3];  // v[3 .. 2R]: in all four windows
#pragma unroll
    for (int k = 4; k <= 2 * R; ++k) c = addv(c, v[k]);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = addv(o[q], c);
  }
}

// Halo position h (outside the output core) of the R-halo plane: the top and
// bottom R rows in full, then the R columns on either side of the core rows.
template <int R, class S>
__device__ __forceinline__ void halo_pos_r(int h, int& row, int& col) {
  constexpr int STRIP = R * S::HW;
  if (h < STRIP) {
    row = h / S::HW;
    col = h - row * S::HW;
  } else if (h < 2 * STRIP) {
    h -= STRIP;
    row = R + S::TY + h / S::HW;
    col = h % S::HW;
  } else {
    h -= 2 * STRIP;
    row = R + h / (2 * R);
    const int c = h % (2 * R);
    col = c < R ? c : kTX + c;
  }
}

// Staged positions of a thread on the R-halo plane (its own outputs first):
// shared-memory index (-1: no position).
template <int R, class S>
__device__ __forceinline__ void split_stage_idx(int tid, int sidx[S::NSTG]) {
  const int ox = tid & 31, oy0 = (tid >> 5) * S::NOUT;
#pragma unroll
  for (int i = 0; i < S::NSTG; ++i) {
    int row, col;
    if (i < S::NOUT) {
      row = oy0 + i + R;
      col = ox + R;
    } else {
      const int h = tid + (i - S::NOUT) * kLnccRHThreads;
      if (h < S::NHALO) {
        halo_pos_r<R, S>(h, row, col);
      } else {
        row = -1;
        col = 0;
      }
    }
    sidx[i] = row < 0 ? -1 : row * S::ZS + col;
  }
}

// In-plane offsets of the staged positions for the tile at (x0, y0): -1
// outside the grid (read as zero), -2 no position.
template <int R, class S>
__device__ __forceinline__ void split_stage_off(const Geom& g, int x0, int y0, const int sidx[S::NSTG],
                                                int soff[S::NSTG]) {
#pragma unroll
  for (int i = 0; i < S::NSTG; ++i) {
    soff[i] = -2;
    if (sidx[i] >= 0) {
      const int row = sidx[i] / S::ZS, col = sidx[i] - row * S::ZS;
      const int x = x0 - R + col, y = y0 - R + row;
      soff[i] = ((unsigned)x < (unsigned)g.fW && (unsigned)y < (unsigned)g.fH) ? y * g.fW + x : -1;
    }
  }
}

template <typename FT, int R>
__global__ void __launch_bounds__(kLnccRHThreads, FFDP_LNCC_SPLIT_MINB) k_lncc_fw(const LnccArgs a) {
  using S = LTS<R>;
  constexpr int W = S::W, TY = S::TY, NOUT = S::NOUT, NSTG = S::NSTG, ZS = S::ZS, HH = S::HH;
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ double wsum[kLnccRHThreads / 32];
  float2* zP = reinterpret_cast<float2*>(sm);
  float2* zQ = zP + HH * ZS;
  float* zX = sm + 4 * HH * ZS;
  constexpr int XS = S::XS, XSX = S::XSX, RB = S::RB;
  float2* xP = reinterpret_cast<float2*>(sm + S::FW_Z);
  float2* xQ = xP + HH * XS;
  float* xX = sm + S::FW_Z + 4 * HH * XS;

  const Geom& g = a.g;
  const int tid = threadIdx.x;
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const float inv_n = a.inv_n, eps = a.eps, gs = a.gscale;
  const float2 ninv2 = make_float2(-inv_n, -inv_n);
  const size_t plane = (size_t)g.fW * g.fH, N = (size_t)g.N;
  float cc_acc = 0.0f;
  if ((tid & 31) == 0) wsum[tid >> 5] = 0.0;
  const int ox = tid & 31, oy0 = (tid >> 5) * NOUT;
  int sidx[NSTG], soff[NSTG];
  split_stage_idx<R, S>(tid, sidx);
  float2 hist[W][NSTG];
  float2 nxt[NSTG];
  auto load_plane = [&](int zp) {
    const bool zin = zp >= 0 && zp < g.fD;
    const size_t base = (size_t)zp * plane;
#pragma unroll
    for (int i = 0; i < NSTG; ++i) {
      float2 v = make_float2(0.0f, 0.0f);
      if (zin && soff[i] >= 0) {
        v.x = ld_stream(a.J + base + soff[i]);
        v.y = ld_stream(F + base + soff[i]);
      }
      nxt[i] = v;
    }
  };

  SegsFw seg(a);
  int tx, ty, z0, z1;
  while (seg.next(tx, ty, z0, z1)) {
    const int x0 = tx * kTX, y0 = ty * TY;
    const int nsteps = (z1 - z0) + 2 * R;
    split_stage_off<R, S>(g, x0, y0, sidx, soff);
    load_plane(z0 - R);
    for (int s0 = 0; s0 < nsteps; s0 += W) {
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int s = s0 + j;
        if (s < nsteps) {
          const int zi = z0 - R + s;  // newest plane; outputs at zc = zi - R
          const bool out = s >= 2 * R;
#pragma unroll
          for (int i = 0; i < NSTG; ++i) hist[j][i] = nxt[i];
          if (s + 1 < nsteps) load_plane(zi + 1);
          if (out) {
            // z sums over the register history -> halo plane
#pragma unroll
            for (int i = 0; i < NSTG; ++i) {
              if (sidx[i] >= 0) {
                float2 sP = hist[0][i];
                float2 sQ = mul2(hist[0][i], hist[0][i]);
                float sX = hist[0][i].x * hist[0][i].y;
#pragma unroll
                for (int q = 1; q < W; ++q) {
                  sP = add2(sP, hist[q][i]);
                  sQ = fma2(hist[q][i], hist[q][i], sQ);
                  sX = fmaf(hist[q][i].x, hist[q][i].y, sX);
                }
                zP[sidx[i]] = sP;
                zQ[sidx[i]] = sQ;
                zX[sidx[i]] = sX;
              }
            }
          }
          __syncthreads();
          if (out) {
            // x sums onto the 32 output columns of every halo row, 4 per item
            // (one channel pair at a time, to bound the live values)
            constexpr int NI = 4 + 2 * R;
            const int row = tid % RB, g4 = tid / RB;
            if (g4 < S::XG4 && row < HH) {
              auto pair4 = [&](const float2* src, float2* dst) {
                const float4* s4 = reinterpret_cast<const float4*>(src + row * ZS + 4 * g4);
                float2 v[NI];
#pragma unroll
                for (int k = 0; k < NI / 2; ++k) {
                  const float4 p = s4[k];
                  v[2 * k] = make_float2(p.x, p.y);
                  v[2 * k + 1] = make_float2(p.z, p.w);
                }
                float2 o[4];
                win4<R>(v, o);
                float4* d4 = reinterpret_cast<float4*>(dst + row * XS + 4 * g4);
                d4[0] = make_float4(o[0].x, o[0].y, o[1].x, o[1].y);
                d4[1] = make_float4(o[2].x, o[2].y, o[3].x, o[3].y);
              };
              pair4(zP, xP);
              pair4(zQ, xQ);
              const float2* s2 = reinterpret_cast<const float2*>(zX + row * ZS + 4 * g4);
              float v[NI];
#pragma unroll
              for (int k = 0; k < NI / 2; ++k) {
                const float2 x = s2[k];
                v[2 * k] = x.x;
                v[2 * k + 1] = x.y;
              }
              float o[4];
              win4<R>(v, o);
              *reinterpret_cast<float4*>(xX + row * XSX + 4 * g4) = make_float4(o[0], o[1], o[2], o[3]);
            }
          }
          __syncthreads();
          if (out) {
            // y sums at the thread's own outputs, cc and the g-terms
            const int zc = zi - R;
            float2 vP[NOUT + 2 * R], vQ[NOUT + 2 * R];
            float vX[NOUT + 2 * R];
#pragma unroll
            for (int k = 0; k < NOUT + 2 * R; ++k) {
              vP[k] = xP[(oy0 + k) * XS + ox];
              vQ[k] = xQ[(oy0 + k) * XS + ox];
              vX[k] = xX[(oy0 + k) * XSX + ox];
            }
            // window sums at the NOUT outputs: the rows shared by all of them
            // once, then each output's own (no sliding; see win4)
            float2 cP = vP[NOUT - 1], cQ = vQ[NOUT - 1];
            float cX = vX[NOUT - 1];
#pragma unroll
            for (int k = NOUT; k <= 2 * R; ++k) {
              cP = add2(cP, vP[k]);
              cQ = add2(cQ, vQ[k]);
              cX += vX[k];
            }
            const int X = x0 + ox;
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              float2 aP = cP, aQ = cQ;
              float aX = cX;
#pragma unroll
              for (int r = k; r < k + 2 * R + 1; ++r) {
                if (r < NOUT - 1 || r > 2 * R) {
                  aP = add2(aP, vP[r]);
                  aQ = add2(aQ, vQ[r]);
                  aX += vX[r];
                }
              }
              const int Y = y0 + oy0 + k;
              if (X < g.fW && Y < g.fH) {
                // aP = (S_J, S_F), aQ = (S_JJ, S_FF), aX = S_FJ; variances clamped at 0
                float2 v = fma2(mul2(aP, aP), ninv2, aQ);
                v = make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f));
                const float cross = fmaf(-aP.x * aP.y, inv_n, aX);
                const float rD = rcp_approx(fmaf(v.x, v.y, eps));
                const float A1 = 2.0f * cross * rD;
                const float cc = cross * cross * rD;
                const float A2 = cc * v.y * rD;
                const size_t lin = ((size_t)zc * g.fH + Y) * g.fW + X;
                a.gbuf[lin] = gs * (2.0f * A2 * aP.x - A1 * aP.y) * inv_n;
                a.gbuf[N + lin] = -gs * A2;
                a.gbuf[2 * N + lin] = gs * A1;
                cc_acc += cc;
              }
            }
          }
          if ((s & 31) == 31) {
            const float v = warp_sum(cc_acc);
            if ((tid & 31) == 0) wsum[tid >> 5] += (double)v;
            cc_acc = 0.0f;
          }
        }
      }
    }
  }
  {
    const float v = warp_sum(cc_acc);
    if ((tid & 31) == 0) wsum[tid >> 5] += (double)v;
  }
  __syncthreads();
  if (tid < kPartialStride) {
    double t = 0.0;
    if (tid == kPCC)
      for (int k = 0; k < kLnccRHThreads / 32; ++k) t += wsum[k];
    a.partials[(size_t)blockIdx.x * kPartialStride + tid] = t;
  }
}

template <typename FT, int BMAX, int R, bool DU>
__global__ void __launch_bounds__(kLnccRHThreads, FFDP_LNCC_SPLIT_MINB) k_lncc_bw(const LnccArgs a) {
  using S = LTS<R>;
  constexpr int W = S::W, TY = S::TY, NOUT = S::NOUT, NSTG = S::NSTG, ZS = S::ZS, HH = S::HH;
  constexpr int XS = S::XS, XSX = S::XSX;
  constexpr bool MI = BMAX != 0;
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ double wsum[kLnccRHThreads / 32][13];
  float2* gP = reinterpret_cast<float2*>(sm);  // (g_J, g_JJ) on the halo plane
  float* gX = sm + 2 * HH * ZS;                 // g_FJ
  float2* gxP = reinterpret_cast<float2*>(sm + S::BW_G);
  float* gxX = sm + S::BW_G + 2 * HH * XS;
  float* slope = sm + S::BW_TOTAL;  // LN_DU: three staging slots of an output plane's slope

  const Geom& g = a.g;
  const int tid = threadIdx.x;
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const size_t plane = (size_t)g.fW * g.fH, N = (size_t)g.N;
  if ((tid & 31) == 0)
    for (int q = 0; q < 13; ++q) wsum[tid >> 5][q] = 0.0;
  DuAcc<NOUT> dacc;
  dacc.clear();
  const int ox = tid & 31, oy0 = (tid >> 5) * NOUT;
  int sidx[NSTG], soff[NSTG];
  split_stage_idx<R, S>(tid, sidx);
  float2 grP[W][NOUT];  // 2-D window sums of the g-terms at the own outputs, last w planes
  float grX[W][NOUT];
  float2 nP[NSTG];      // next g plane at the staged positions
  float nX[NSTG];
  float2 jf[NOUT], jfn[NOUT];  // (J, F) at the own outputs of this and of the next output plane
  auto load_g = [&](int zp) {
    const bool zin = zp >= 0 && zp < g.fD;
    const size_t base = (size_t)zp * plane;
#pragma unroll
    for (int i = 0; i < NSTG; ++i) {
      float2 v = make_float2(0.0f, 0.0f);
      float x = 0.0f;
      if (zin && soff[i] >= 0) {
        const float* p = a.gbuf + base + soff[i];
        v.x = ld_stream(p);
        v.y = ld_stream(p + N);
        x = ld_stream(p + 2 * N);
      }
      nP[i] = v;
      nX[i] = x;
    }
  };

  SegsBw seg(a);
  int tx, ty, z0, z1;
  while (seg.next(tx, ty, z0, z1)) {
    const int x0 = tx * kTX, y0 = ty * TY;
    const int nsteps = (z1 - z0) + 2 * R;
    const bool full = x0 + kTX <= g.fW && y0 + TY <= g.fH && (g.fW & 3) == 0;
    const size_t slope_plane = 3 * (size_t)g.fW * g.fH;
    const float* slope_tile = DU ? a.dJdq + 3 * ((size_t)y0 * g.fW + x0) : nullptr;
    int slot_rd = 2;
    auto fold_du = [&] {
      float cy[NOUT];
#pragma unroll
      for (int k = 0; k < NOUT; ++k) cy[k] = (float)(y0 + oy0 + k) - g.ctr[1];
      dacc.fold(wsum[tid >> 5], tid & 31, (float)(x0 + ox) - g.ctr[0], cy);
    };
    // (J, F) at the own outputs of output plane zo (zero outside the grid)
    auto load_jf = [&](int zo) {
      const int X = x0 + ox;
#pragma unroll
      for (int k = 0; k < NOUT; ++k) {
        const int Y = y0 + oy0 + k;
        float2 v = make_float2(0.0f, 0.0f);
        if (zo >= 0 && zo < g.fD && X < g.fW && Y < g.fH) {
          const size_t lin = ((size_t)zo * g.fH + Y) * g.fW + X;
          v.x = ld_stream(a.J + lin);
          v.y = ld_stream(F + lin);
        }
        jfn[k] = v;
      }
    };
    split_stage_off<R, S>(g, x0, y0, sidx, soff);
    load_g(z0 - R);
    for (int s0 = 0; s0 < nsteps; s0 += W) {
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int s = s0 + j;
        if (s < nsteps) {
          const int zi = z0 - R + s;  // newest g plane; outputs at zo = zi - R
          // the fetched plane goes to the halo plane; fetch the next, and the
          // (J, F) and slope of the next step's output plane
#pragma unroll
          for (int i = 0; i < NSTG; ++i) {
            if (sidx[i] >= 0) {
              gP[sidx[i]] = nP[i];
              gX[sidx[i]] = nX[i];
            }
          }
#pragma unroll
          for (int k = 0; k < NOUT; ++k) jf[k] = jfn[k];
          if (s + 1 < nsteps) load_g(zi + 1);
          if (s + 1 >= 2 * R && s + 1 < nsteps) load_jf(zi + 1 - R);
          if constexpr (DU) {
            slot_rd = slot_rd == 2 ? 0 : slot_rd + 1;
            const int sn = s + 1;
            const float* src =
                (sn >= 2 * R && sn < nsteps) ? slope_tile + (size_t)(zi + 1 - R) * slope_plane : nullptr;
            stage_slope<TY, kLnccRHThreads>(slope + (slot_rd == 2 ? 0 : slot_rd + 1) * SlopeStage<TY>::SLOT, src,
                                            g, x0, y0, full, tid);
            slope_wait_prev();
          }
          __syncthreads();
          {
            // x sums of the g-terms onto the 32 output columns, 2 per item
            constexpr int NI = 2 + 2 * R;
            for (int it = tid; it < HH * (kTX / 2); it += kLnccRHThreads) {
              const int row = it / (kTX / 2), g2 = it - row * (kTX / 2);
              const float4* s4 = reinterpret_cast<const float4*>(gP + row * ZS + 2 * g2);
              const float2* s2 = reinterpret_cast<const float2*>(gX + row * ZS + 2 * g2);
              float2 vP[NI];
              float vX[NI];
#pragma unroll
              for (int k = 0; k < NI / 2; ++k) {
                const float4 p = s4[k];
                const float2 x = s2[k];
                vP[2 * k] = make_float2(p.x, p.y);
                vP[2 * k + 1] = make_float2(p.z, p.w);
                vX[2 * k] = x.x;
                vX[2 * k + 1] = x.y;
              }
              float2 cP = vP[1];
              float cX = vX[1];
#pragma unroll
              for (int k = 2; k <= 2 * R; ++k) {
                cP = add2(cP, vP[k]);
                cX += vX[k];
              }
              const float2 aP = add2(vP[0], cP), bP = add2(cP, vP[2 * R + 1]);
              *reinterpret_cast<float4*>(gxP + row * XS + 2 * g2) = make_float4(aP.x, aP.y, bP.x, bP.y);
              *reinterpret_cast<float2*>(gxX + row * XSX + 2 * g2) = make_float2(vX[0] + cX, cX + vX[2 * R + 1]);
            }
          }
          __syncthreads();
          {
            // y sums at the own outputs -> register ring slot j
            float2 vP[NOUT + 2 * R];
            float vX[NOUT + 2 * R];
#pragma unroll
            for (int k = 0; k < NOUT + 2 * R; ++k) {
              vP[k] = gxP[(oy0 + k) * XS + ox];
              vX[k] = gxX[(oy0 + k) * XSX + ox];
            }
            // the rows shared by all NOUT outputs once, then each output's own
            float2 cP = vP[NOUT - 1];
            float cX = vX[NOUT - 1];
#pragma unroll
            for (int k = NOUT; k <= 2 * R; ++k) {
              cP = add2(cP, vP[k]);
              cX += vX[k];
            }
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              float2 aP = cP;
              float aX = cX;
#pragma unroll
              for (int r = k; r < k + 2 * R + 1; ++r) {
                if (r < NOUT - 1 || r > 2 * R) {
                  aP = add2(aP, vP[r]);
                  aX += vX[r];
                }
              }
              grP[j][k] = aP;
              grX[j][k] = aX;
            }
          }
          // z sums over the ring (the w planes zo - R .. zo + R) -> dL/dJ at zo
          if (s >= 2 * R) {
            const int zo = zi - R;
#pragma unroll
            for (int k = 0; k < NOUT; ++k) {
              float2 bP = grP[0][k];
              float bX = grX[0][k];
#pragma unroll
              for (int q = 1; q < W; ++q) {
                bP = add2(bP, grP[q][k]);
                bX += grX[q][k];
              }
              const int X = x0 + ox, Y = y0 + oy0 + k;
              if (X < g.fW && Y < g.fH) {
                const size_t lin = ((size_t)zo * g.fH + Y) * g.fW + X;
                const float jv = jf[k].x, fv = jf[k].y;
                float gv = fmaf(fv, bX, fmaf(2.0f * jv, bP.y, bP.x));
                if (MI) gv += mi_grad_ln<(MI ? BMAX : 32)>(a.T, a.bf, a.bj, fv, jv);
                if constexpr (DU) {
                  dacc.add(a, k, lin, slope + slot_rd * SlopeStage<TY>::SLOT + (oy0 + k) * SlopeStage<TY>::ROW + 3 * ox,
                           (float)zo - g.ctr[2], gv);
                } else if (a.dJ) {
                  a.dJ[lin] = gv;
                }
              }
            }
          }
          if constexpr (DU) {
            if ((s & 31) == 31) fold_du();
          }
        }
      }
    }
    if constexpr (DU) fold_du();  // the next segment has other columns and rows
  }
  if constexpr (DU) {
    __syncthreads();
    if (tid < 12) {
      double t = 0.0;
      for (int k = 0; k < kLnccRHThreads / 32; ++k) t += wsum[k][tid];
      a.partials[(size_t)blockIdx.x * kPartialStride + tid] = t;
    }
  }
}

template <int R, bool DU>
static size_t smem_of() {
  const size_t stage = (DU && !kLnccRecompute) ? (size_t)SlopeStage<LT<R>::TY>::FLOATS : 0;
  return ((size_t)LTR<R>::TOTAL + stage) * sizeof(float);
}

// occ != nullptr: report resident CTAs per SM instead of launching.
template <typename FT, int BMAX, int R, bool DU>
static cudaError_t run_lncc(const LnccArgs& a, int grid, cudaStream_t s, int* occ) {
  auto k = k_lncc_rh<FT, BMAX, R, DU>;
  const size_t smem = smem_of<R, DU>();
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int nt = kLnccRHThreads;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, nt, smem);
  note_launch_begin("k_lncc", s);
  k<<<grid, nt, smem, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

// Split variant: the forward and the backward kernel on the same grid (the
// forward one writes every CTA's whole partial record, the backward one adds
// the affine slots).  occ != nullptr: the smaller of their occupancies.
template <typename FT, int BMAX, int R, bool DU>
static cudaError_t run_split(const LnccArgs& a, int grid, cudaStream_t s, int* occ) {
  auto k1 = k_lncc_fw<FT, R>;
  auto k2 = k_lncc_bw<FT, BMAX, R, DU>;
  const size_t m1 = (size_t)LTS<R>::FW_TOTAL * sizeof(float);
  const size_t m2 = ((size_t)LTS<R>::BW_TOTAL + (DU ? (size_t)SlopeStage<LTS<R>::TY>::FLOATS : 0)) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m1);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m2);
  if (e != cudaSuccess) return e;
  if (occ) {
    int o1 = 0, o2 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, k1, kLnccRHThreads, m1);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, k2, kLnccRHThreads, m2);
    *occ = o1 < o2 ? o1 : o2;
    return e;
  }
  note_launch_begin("k_lncc_fw", s);
  k1<<<grid, kLnccRHThreads, m1, s>>>(a);
  note_launch_end(s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch_begin("k_lncc_bw", s);
  k2<<<grid, kLnccRHThreads, m2, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

template <typename FT, int BMAX, int R, bool DU>
static cudaError_t run_any(const LnccArgs& a, int grid, cudaStream_t s, int* occ) {
  if constexpr (kLnccSplit && !kLnccRecompute)
    return run_split<FT, BMAX, R, DU>(a, grid, s, occ);
  else
    return run_lncc<FT, BMAX, R, DU>(a, grid, s, occ);
}

template <int R>
static cudaError_t dispatch_r(int mode, int ft, int bmax, const LnccArgs& a, int grid, cudaStream_t s, int* occ) {
  // LN_DJ (the stand-alone LNCC gradient) carries no MI term; LN_DU (the
  // objective) any bin count
  cudaError_t e = cudaErrorInvalidValue;
  if (mode == LN_DJ && bmax != 0) return e;
  FFDP_DT_SWITCH(ft, FT, {
    if (mode == LN_DJ)
      e = run_any<FT, 0, R, false>(a, grid, s, occ);
    else if (bmax == 0)
      e = run_any<FT, 0, R, true>(a, grid, s, occ);
    else if (bmax == 32)
      e = run_any<FT, 32, R, true>(a, grid, s, occ);
    else
      e = run_any<FT, 64, R, true>(a, grid, s, occ);
  });
  return e;
}

static cudaError_t dispatch_lncc(int mode, int ft, int mt, int bmax, const LnccArgs& a, int grid,
                                 cudaStream_t s, int R, int* occ) {
  switch (R) {
    case 1: return dispatch_r<1>(mode, ft, bmax, a, grid, s, occ);
    case 2: return dispatch_r<2>(mode, ft, bmax, a, grid, s, occ);
    case 3: return dispatch_r<3>(mode, ft, bmax, a, grid, s, occ);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_lncc(int mode, int ft, int mt, int bmax, const LnccArgs& a, int grid, cudaStream_t s) {
  return dispatch_lncc(mode, ft, mt, bmax, a, grid, s, a.R, nullptr);
}

int lncc_ctas_per_sm(int mode, int ft, int mt, int bmax, int R) {
  static OccCache<2 * 2 * 3 * 4> cache;
  const int bidx = bmax == 0 ? 0 : (bmax == 32 ? 1 : 2);
  return cache.get(((mode * 2 + ft) * 3 + bidx) * 4 + (R >= 0 && R <= 3 ? R : 0), [&] {
    int occ = 0;
    LnccArgs dummy{};
    return dispatch_lncc(mode, ft, mt, bmax, dummy, 0, 0, R, &occ) == cudaSuccess ? occ : 1;
  });
}

}  // namespace ffdp
