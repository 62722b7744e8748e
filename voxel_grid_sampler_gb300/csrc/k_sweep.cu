// k_sweep.cu -- voxel-linear sweeps of the fused objective.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration".  Key designs item 1: the composite implicit grid sampler
// I(Ax+t+Su(x)) and its backward (with the affine gradient) run with every
// coordinate in registers.  Key designs item 2: Mattes MI through an implicit
// Parzen window -- histogram entries accumulate per voxel in shared memory and
// the per-voxel partial gradient reads a small table, so no B x N block exists.
//
// Layout of the work: a CTA iteration covers (CTA threads)*kVPT consecutive
// voxels of the flattened [D][H][W] grid; each warp owns 32*kVPT of them and
// each lane every 32nd (see the lane walk), taken two at a time through a
// two-stage gather pipeline.  Grids are persistent (one CTA per SM striding
// over iterations).
#include "ffdp_internal.h"

namespace ffdp {

// ----------------------------------------------------- histogram layout
// Shared atomic instructions of a warp are conflict-free by construction:
//
// * BMAX = 32: every lane owns a private copy of the joint histogram, word
//   (a * 32 + b) * 32 + lane; all 32 lanes of an instruction hit 32 banks and
//   the 16 words of a voxel sit at compile-time offsets from one base.
// * BMAX = 64 (a private copy per lane would not fit): R = 8 lane copies per
//   bin.  Lane l adds into copy c = l mod 8, and its group ga = l / 8 (0..3)
//   fixes the order in which it visits a voxel's four kernel rows: at step i
//   the row a of the four with a = i + ga (mod 4).  The word address
//     word(a, b, c) = (a / 4) * 32 B + 32 b + 8 (a mod 4) + c
//   lies in bank 8 (a mod 4) + c, so at every step the 32 lanes use 32
//   distinct banks whatever their bins.
template <int BMAX>
struct HistLayout {
  static constexpr bool PRIVATE = BMAX <= 32;
  static constexpr int R = PRIVATE ? 32 : 8;      // copies per bin
  static constexpr int COL = PRIVATE ? 32 : 4 * R;  // word stride of b
  static constexpr int QROW = COL * BMAX;         // words per row (private) / per group of four rows
  static constexpr int WORDS = BMAX * BMAX * R;
  __host__ __device__ static constexpr int word(int a, int b) {
    return PRIVATE ? (a * BMAX + b) * 32 : (a >> 2) * QROW + COL * b + R * (a & 3);
  }
};

// u32 fixed-point counts (kHistFrac fraction bits): one voxel adds at most
// (2/3)^2 to a word, so a CTA flushes its copies to the u64 global histogram
// at least every flush_every<BMAX, NT>() iterations.
// A CTA of NT threads adds at most NT * kVPT / R voxels to one word per iteration.
template <int BMAX, int NT>
__host__ __device__ constexpr int flush_every() {
  return (int)(4294967295.0 / ((double)NT * kVPT / HistLayout<BMAX>::R * (4.0 / 9.0) * kHistOne)) - 1;
}
static_assert(flush_every<32, kSweep1Threads>() >= 16 && flush_every<64, kSweep1Threads>() >= 16,
              "histogram flush interval");

// fp32 per-thread gradient partials are folded into fp64 every this many iterations.
constexpr int kFoldEvery = 16;

__global__ void k_zero_u64(unsigned long long* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0ull;
}

// Sums the R copies of every bin into the u64 histogram and clears them.
// Private copies: a thread reads the 32 words of its bin starting at its own
// lane's bank.  Shared copies: thread i reads bin (a, b) with a mod 4 = i mod 4
// and takes its two 16-byte halves in lane-dependent order, so the 8 lanes of
// each quarter-warp read 8 different bank quads (rows run to B rounded up to
// a multiple of 4).
template <int BMAX, int NT>
__device__ __forceinline__ void hist_flush(unsigned* hist, unsigned long long* gh, int B) {
  using L = HistLayout<BMAX>;
  __syncthreads();
  if (L::PRIVATE) {
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < B * B; i += NT) {
      const int ra = i / B, rb = i - ra * B;
      unsigned* w = hist + L::word(ra, rb);
      unsigned long long s = 0ull;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) {
        const int c = (lane + j) & 31;
        s += w[c];
        w[c] = 0u;
      }
      if (s) atomicAdd(gh + i, s);
    }
  } else {
    static_assert(L::PRIVATE || L::R == 8, "flush reads two uint4 per bin");
    const int h = (threadIdx.x >> 2) & 1;
    const int n = ((B + 3) & ~3) * B;
    for (int i = threadIdx.x; i < n; i += NT) {
      const int rest = i >> 2, rb = rest % B, ra = ((rest / B) << 2) | (i & 3);
      if (ra >= B) continue;
      uint4* w = reinterpret_cast<uint4*>(hist + L::word(ra, rb));
      const uint4 v0 = w[h], v1 = w[h ^ 1];
      w[h] = make_uint4(0u, 0u, 0u, 0u);
      w[h ^ 1] = make_uint4(0u, 0u, 0u, 0u);
      const unsigned long long s = (unsigned long long)v0.x + v0.y + (unsigned long long)v0.z + v0.w +
                                   (unsigned long long)v1.x + v1.y + (unsigned long long)v1.z + v1.w;
      if (s) atomicAdd(gh + ra * B + rb, s);
    }
  }
  __syncthreads();
}

// Per-lane constants of the histogram accumulation.
struct HistLane {
  int rowoff[4];  // shared copies: R ((i + ga) mod 4) + c for step i; private: lane
  int ga;
};

template <int BMAX>
__device__ __forceinline__ void hist_lane_init(HistLane& h) {
  using L = HistLayout<BMAX>;
  const int lane = threadIdx.x & 31;
  h.ga = lane / 8;
#pragma unroll
  for (int i = 0; i < 4; ++i) h.rowoff[i] = L::PRIVATE ? lane : 8 * ((i + h.ga) & 3) + (lane & 7);
}

// r[i] = w[(i + s) mod 4].
__device__ __forceinline__ void rotate4(const float w[4], int s, float r[4]) {
  const bool s1 = (s & 1) != 0, s2 = (s & 2) != 0;
  float t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = s1 ? w[(i + 1) & 3] : w[i];
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = s2 ? t[(i + 2) & 3] : t[i];
}

// Parzen contribution of one voxel: beta(a - cF) beta(b - cJ) on the 4x4 bins
// around (cF, cJ), rounded to fixed point by the multiply itself: the F
// weights carry 2^-65 and the J weights 2^-64 (both stay normal floats), so
// their product beta beta' 2^-129 = (beta beta' 2^kHistFrac) 2^-149 is a
// subnormal float whose bit pattern is that count rounded to nearest even --
// one multiply per bin, no conversion (device code keeps subnormals: no
// flush-to-zero).
template <int BMAX>
__device__ __forceinline__ void hist_add(unsigned* hist, const HistLane& h, const BinMap& bf, const BinMap& bj,
                                         float f, float j) {
  using L = HistLayout<BMAX>;
  int af, aj;
  float tf, tj;
  floor_split(bin_coord(bf, f), af, tf);
  floor_split(bin_coord(bj, j), aj, tj);
  float wf[4], wj[4];
  bspline4(tf, kHistScaleF, wf);
  bspline4(tj, kHistScaleJ, wj);
  if (L::PRIVATE) {
    unsigned* base = hist + L::word(af - 1, aj - 1) + h.rowoff[0];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        atomicAdd(base + i * L::QROW + k * L::COL, __float_as_uint(__fmul_rn(wf[i], wj[k])));
  } else {
    // step i takes kernel row a_i = af - 1 + ((i + s) mod 4), s = ga - af + 1,
    // so that a_i = i + ga (mod 4)
    const int s = h.ga - af + 1;
    float wr[4];
    rotate4(wf, s, wr);
    unsigned* col = hist + L::COL * (aj - 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ai = af - 1 + ((i + s) & 3);
      unsigned* row = col + (ai >> 2) * L::QROW + h.rowoff[i];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        atomicAdd(row + k * L::COL, __float_as_uint(__fmul_rn(wr[i], wj[k])));
    }
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

// ------------------------------------------------------------- lane walk
// Lane l of warp w handles, in CTA iteration it, the voxels
//   lin = it * NT * kVPT + w * 32 * kVPT + l + 32 v,  v = 0..kVPT-1  (NT threads per CTA).
// Every load, gather and store instruction of a warp covers 32 consecutive
// voxels, so F, J, g and dJ move in whole 128-byte lines and the trilinear
// taps of 32 neighbouring points share one or two lines per M row.
struct LaneWalk {
  long long P[3];  // fixed-point anchor G i + g0 of the current voxel
  int x, y, z;
};

__device__ __forceinline__ void lw_seek(const Geom& g, unsigned lin, LaneWalk& w) {
  lin_to_xyz(g, lin, w.x, w.y, w.z);
  anchor(g, w.x, w.y, w.z, w.P);
}

// Moves to voxel lin = previous + 32: inside the row the anchor advances by
// the exact fixed-point step 32 G e_x, otherwise it is recomputed.
__device__ __forceinline__ void lw_step(const Geom& g, unsigned lin, LaneWalk& w) {
  if (w.x + 32 < g.fW) {
    w.x += 32;
    w.P[0] += g.Gq[0] * 32;
    if (!g.a_diag) {
      w.P[1] += g.Gq[3] * 32;
      w.P[2] += g.Gq[6] * 32;
    }
  } else {
    lw_seek(g, lin, w);
  }
}

// Number of the lane's kVPT voxels (32 apart from lin0) inside the grid.
__device__ __forceinline__ int lane_count(unsigned lin0, unsigned N) {
  return lin0 >= N ? 0 : min((int)((N - lin0 + 31u) >> 5), kVPT);
}

// ------------------------------------------------------ streamed inputs
// The per-voxel inputs of a warp's chunk of 32*kVPT voxels (u: 12 B, F: 2 or
// 4 B, J or g: 4 B per voxel) reach shared memory through 1-D bulk
// asynchronous copies that lane 0 of the warp issues NST chunks ahead into a
// per-warp ring of NST slots; each slot's completion is counted in bytes on
// its own mbarrier.  HBM therefore always holds several chunks per warp in
// flight, independent of the warp's instruction stream.  Only whole chunks
// are streamed; the one ragged chunk at the end of the grid is read directly.

// Set when a bounded wait for a ring slot gave up; outputs of that call are
// invalid (the finish kernel then writes NaN losses).
__device__ unsigned g_ffdp_device_error;

constexpr unsigned long long kWaitNs = 1000000000ull;  // a ring wait gives up after 1 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the completion of phase `parity`; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitNs) return false;
  return true;
}

// Streamed inputs are read once: mark them first for eviction from L2, which
// keeps the randomly gathered moving image resident.
__device__ __forceinline__ unsigned long long policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, unsigned bytes, uint32_t bar,
                                         unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Ring geometry: per slot [u][F][X] for one chunk; NST slots per warp, then
// one 8-byte mbarrier per slot after all warps' slots.
template <typename FT, bool SU, bool SF, bool SX, int NST, int NT>
struct Ring {
  static constexpr int kChunk = 32 * kVPT;
  static constexpr int kU = SU ? kChunk * 12 : 0;
  static constexpr int kF = SF ? kChunk * (int)sizeof(FT) : 0;
  static constexpr int kX = SX ? kChunk * 4 : 0;
  static constexpr int kSlot = kU + kF + kX;
  static constexpr int kWarps = NT / 32;
  static constexpr size_t kBytes = (size_t)kWarps * NST * (kSlot + 8);
  static_assert(kU % 16 == 0 && kF % 16 == 0 && kX % 16 == 0, "bulk copies move multiples of 16 bytes");
};

// Per-warp view of the ring.
template <class RG, int NST>
struct WarpRing {
  using RGT = RG;
  char* slots;    // this warp's NST slots
  uint32_t bars;  // shared address of this warp's first mbarrier
  unsigned tx;    // bytes per chunk (0: nothing streamed)
  bool has_u;

  __device__ __forceinline__ void init(char* ring, bool has_u_) {
    const int warp = threadIdx.x >> 5;
    slots = ring + (size_t)warp * NST * RG::kSlot;
    bars = smem_u32(ring + (size_t)RG::kWarps * NST * RG::kSlot) + warp * NST * 8;
    has_u = has_u_ && RG::kU > 0;
    tx = (has_u ? RG::kU : 0) + RG::kF + RG::kX;
    if (tx && (threadIdx.x & 31) == 0) {
#pragma unroll
      for (int s = 0; s < NST; ++s) mbar_init(bars + 8 * s, 1);
      mbar_fence_init();
    }
    __syncwarp();
  }

  // lane 0: copy chunk ch into slot s (the barrier expects `extra` bytes more
  // than the copies deliver when a test arms a stall)
  template <typename FT>
  __device__ __forceinline__ void issue(int s, unsigned ch, const float* u, const FT* F, const float* X,
                                        unsigned long long pol, unsigned extra = 0) const {
    const size_t v0 = (size_t)ch * RG::kChunk;
    char* slot = slots + s * RG::kSlot;
    const uint32_t bar = bars + 8 * s;
    mbar_expect_tx(bar, tx + extra);
    if (RG::kU && has_u) bulk_g2s(smem_u32(slot), u + 3 * v0, RG::kU, bar, pol);
    if (RG::kF) bulk_g2s(smem_u32(slot + RG::kU), F + v0, RG::kF, bar, pol);
    if (RG::kX) bulk_g2s(smem_u32(slot + RG::kU + RG::kF), X + v0, RG::kX, bar, pol);
  }

  __device__ __forceinline__ const float* u_of(int s) const { return reinterpret_cast<const float*>(slots + s * RG::kSlot); }
  template <typename FT>
  __device__ __forceinline__ const FT* f_of(int s) const {
    return reinterpret_cast<const FT*>(slots + s * RG::kSlot + RG::kU);
  }
  __device__ __forceinline__ const float* x_of(int s) const {
    return reinterpret_cast<const float*>(slots + s * RG::kSlot + RG::kU + RG::kF);
  }
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }

// The ring schedule of one warp: iteration k of the CTA loop (it = blockIdx.x
// + k gridDim.x) takes chunk it * kWarps + warp from slot k mod NST, whose
// (k / NST)-th completion has parity (k / NST) & 1.  A wait that gives up
// sets the device error word; the warp then stops streaming (its later
// chunks read nothing) and, before exiting, waits (bounded) for the copies it
// still has in flight.
template <class WR, int NST>
struct RingSched {
  unsigned nIter, nFull;  // CTA iterations; whole chunks in the grid
  int kfail;              // first iteration whose wait gave up (-1: none)

  __device__ __forceinline__ unsigned chunk(unsigned it) const { return it * WR::RGT::kWarps + (threadIdx.x >> 5); }
  __device__ __forceinline__ bool streamed(unsigned it) const { return it < nIter && chunk(it) < nFull; }

  // stall_tx != 0 (tests only): slot 0 expects that many bytes more than its
  // copies deliver, so every wait on it runs out.
  template <typename FT>
  __device__ __forceinline__ void prologue(const WR& r, const float* u, const FT* F, const float* X,
                                           unsigned long long pol, unsigned stall_tx = 0) const {
    if (r.tx != 0 && (threadIdx.x & 31) == 0) {
#pragma unroll
      for (int s = 0; s < NST; ++s) {
        const unsigned it = blockIdx.x + s * gridDim.x;
        if (streamed(it)) r.template issue<FT>(s, chunk(it), u, F, X, pol, s == 0 ? stall_tx : 0u);
      }
    }
    __syncwarp();
  }

  // Waits for slot k mod NST; false (uniform over the warp) if it gave up.
  __device__ __forceinline__ bool wait(const WR& r, unsigned k) {
    if (kfail >= 0) return false;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(r.bars + 8 * (k % NST), (k / NST) & 1));
    if (!ok) {
      kfail = (int)k;
      if ((threadIdx.x & 31) == 0) atomicExch(&g_ffdp_device_error, 1u);
    }
    return ok;
  }

  // After the warp has read slot k mod NST: refill it with the chunk NST iterations ahead.
  template <typename FT>
  __device__ __forceinline__ void refill(const WR& r, unsigned k, unsigned it, const float* u, const FT* F,
                                         const float* X, unsigned long long pol) const {
    __syncwarp();
    const unsigned it2 = it + NST * gridDim.x;
    if (kfail < 0 && (threadIdx.x & 31) == 0 && streamed(it2)) r.template issue<FT>(k % NST, chunk(it2), u, F, X, pol);
    __syncwarp();
  }

  // Bounded drain of the copies still in flight after a failed wait.
  __device__ __forceinline__ void drain(const WR& r) const {
    if (kfail < 0 || (threadIdx.x & 31) != 0) return;
    for (unsigned k = (unsigned)kfail; k < (unsigned)kfail + NST; ++k)
      if (streamed(blockIdx.x + k * gridDim.x)) mbar_wait(r.bars + 8 * (k % NST), (k / NST) & 1);
  }
};

// ------------------------------------------------------ half-chunk pipeline
// A lane's kVPT = 4 voxels of a chunk are taken two at a time ("halves").
// While one half is interpolated and accumulated, the 16 trilinear taps of the
// next half (the second half of this chunk, or the first half of the warp's
// next chunk) are already in flight, so gather latency overlaps arithmetic.
static_assert(kVPT == 4, "the pipeline takes a lane's four voxels as two halves");

struct Half {
  float taps[2][8];
  float rr[2][3];
  float f[2];       // F (histogram / MI)
  float x[2];       // J (MI on a given J) or g = dL/dJ (given gradient)
  int ix[2], iy[2], iz[2];
  unsigned lin;     // linear index of the half's first voxel (this lane)
  int nv;           // voxels of the half inside the grid (0..2)
};

// Prepares half h (0 or 1) of iteration k (CTA iteration it): reads u, F and
// J/g (from the ring slot of a streamed chunk, else from global memory),
// walks the coordinates and issues the gathers.  Half 0 waits for the chunk's
// slot; half 1 releases the slot for refilling.
// LU streams the 3-vector slot (u, or the stored dJ/dq when GATHER is off);
// GATHER walks the fixed-point coordinates and gathers the taps; without it
// the slot's vector is kept in H.rr and only the voxel indices are walked.
// IA: every anchor is an integer (Geom::ia), so the walk keeps voxel indices
// only and the cell comes from cell_of_int (the same cells and fractions).
template <typename FT, typename MT, bool LF, bool LU, bool LX, bool GATHER, bool IA, class WR, int NST>
__device__ __forceinline__ void prepare(Half& H, const Geom& g, const MT* __restrict__ M, const FT* __restrict__ F,
                                        const float* u, const float* X, WR& wr, RingSched<WR, NST>& rs,
                                        LaneWalk& w, unsigned it, unsigned k, int h, unsigned long long pol) {
  const int lane = threadIdx.x & 31;
  const unsigned ch = rs.chunk(it);
  const unsigned lin0 = ch * (32 * kVPT) + lane;
  const int nvc = it < rs.nIter ? lane_count(lin0, g.N) : 0;
  H.lin = lin0 + 64u * h;
  H.nv = min(max(nvc - 2 * h, 0), 2);
  const bool streamed = wr.tx && it < rs.nIter && ch < rs.nFull;
  bool ok = true;
  if (streamed && h == 0) ok = rs.wait(wr, k);
  const int s = k % NST;
  float uu[2][3];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int v = 2 * h + j;
    const unsigned lin = lin0 + 32u * v;
    H.f[j] = H.x[j] = uu[j][0] = uu[j][1] = uu[j][2] = 0.0f;
    if (streamed) {
      if (ok) {
        const int e = lane + 32 * v;
        if (LF) H.f[j] = to_f(wr.template f_of<FT>(s)[e]);
        if (LU && wr.has_u) {
          uu[j][0] = wr.u_of(s)[3 * e + 0];
          uu[j][1] = wr.u_of(s)[3 * e + 1];
          uu[j][2] = wr.u_of(s)[3 * e + 2];
        }
        if (LX) H.x[j] = wr.x_of(s)[e];
      }
    } else if (v < nvc) {
      if (LF) H.f[j] = load1(F + lin);
      if (LU && u) {
        uu[j][0] = __ldg(u + 3ull * lin + 0);
        uu[j][1] = __ldg(u + 3ull * lin + 1);
        uu[j][2] = __ldg(u + 3ull * lin + 2);
      }
      if (LX) H.x[j] = __ldg(X + lin);
    }
  }
  if (streamed && h == 1) rs.template refill<FT>(wr, k, it, u, F, X, pol);
  if (LU && GATHER) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = 2 * h + j;
      int b[3];
      if constexpr (IA) {
        // integer anchors: the walk needs only the voxel indices
        if (v < nvc) {
          if (v > 0 && w.x + 32 < g.fW)
            w.x += 32;
          else
            lin_to_xyz(g, lin0 + 32u * v, w.x, w.y, w.z);
        }
        cell_of_int(g, w.x, w.y, w.z, uu[j][0], uu[j][1], uu[j][2], b, H.rr[j]);
      } else {
        if (v < nvc) {
          if (v == 0)
            lw_seek(g, lin0, w);
          else
            lw_step(g, lin0 + 32u * v, w);
        }
        cell_of(g, w.P, uu[j][0], uu[j][1], uu[j][2], b, H.rr[j]);
      }
      H.ix[j] = w.x;
      H.iy[j] = w.y;
      H.iz[j] = w.z;
      if (v >= nvc) b[0] = -2;  // past the end: no loads
      gather8<MT>(M, g, b, H.taps[j]);
    }
  } else if (LU) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = 2 * h + j;
      if (v < nvc) {
        if (v > 0 && w.x + 32 < g.fW)
          w.x += 32;
        else
          lin_to_xyz(g, lin0 + 32u * v, w.x, w.y, w.z);
      }
      H.ix[j] = w.x;
      H.iy[j] = w.y;
      H.iz[j] = w.z;
      H.rr[j][0] = uu[j][0];
      H.rr[j][1] = uu[j][1];
      H.rr[j][2] = uu[j][2];
    }
  }
}

// Non-gathering passes (streamed J / g and slope): a whole chunk per step,
// one wait, one refill and one coordinate seek for the lane's four voxels.
template <typename FT, bool LF, bool LU, bool LX, class WR, int NST>
__device__ __forceinline__ void prepare_chunk(Half& A, Half& B, const Geom& g, const FT* __restrict__ F,
                                              const float* u, const float* X, WR& wr, RingSched<WR, NST>& rs,
                                              unsigned it, unsigned k, unsigned long long pol) {
  const int lane = threadIdx.x & 31;
  const unsigned ch = rs.chunk(it);
  const unsigned lin0 = ch * (32 * kVPT) + lane;
  const int nvc = it < rs.nIter ? lane_count(lin0, g.N) : 0;
  A.lin = lin0;
  B.lin = lin0 + 64u;
  A.nv = min(nvc, 2);
  B.nv = min(max(nvc - 2, 0), 2);
  const bool streamed = wr.tx && it < rs.nIter && ch < rs.nFull;
  bool ok = true;
  if (streamed) ok = rs.wait(wr, k);
  const int s = k % NST;
  int x = 0, y = 0, z = 0;
  if (nvc > 0) lin_to_xyz(g, lin0, x, y, z);
#pragma unroll
  for (int v = 0; v < kVPT; ++v) {
    Half& H = v < 2 ? A : B;
    const int j = v & 1;
    const unsigned lin = lin0 + 32u * v;
    H.f[j] = H.x[j] = H.rr[j][0] = H.rr[j][1] = H.rr[j][2] = 0.0f;
    if (streamed) {
      if (ok) {
        const int e = lane + 32 * v;
        if (LF) H.f[j] = to_f(wr.template f_of<FT>(s)[e]);
        if (LU && wr.has_u) {
          H.rr[j][0] = wr.u_of(s)[3 * e + 0];
          H.rr[j][1] = wr.u_of(s)[3 * e + 1];
          H.rr[j][2] = wr.u_of(s)[3 * e + 2];
        }
        if (LX) H.x[j] = wr.x_of(s)[e];
      }
    } else if (v < nvc) {
      if (LF) H.f[j] = load1(F + lin);
      if (LU && u) {
        H.rr[j][0] = __ldg(u + 3ull * lin + 0);
        H.rr[j][1] = __ldg(u + 3ull * lin + 1);
        H.rr[j][2] = __ldg(u + 3ull * lin + 2);
      }
      if (LX) H.x[j] = __ldg(X + lin);
    }
    if (v > 0 && v < nvc) {
      if (x + 32 < g.fW)
        x += 32;
      else
        lin_to_xyz(g, lin, x, y, z);
    }
    H.ix[j] = x;
    H.iy[j] = y;
    H.iz[j] = z;
  }
  if (streamed) rs.template refill<FT>(wr, k, it, u, F, X, pol);
}

// ------------------------------------------------------------------ sweep 1
// Sampling (or reading J) plus, per mode, the histogram and/or a J store
// (and, for the LNCC objective, a store of the slope dJ/dq, so that its
// sampler backward streams instead of gathering M again).
// Streams: u (sampling), F (histogram), J (histogram of a given J).
template <typename FT, int BMAX, int MODE>
struct S1Cfg {
  static constexpr bool HIST = MODE != S1_WRITEJ && MODE != S1_WRITEJG;
  static constexpr bool SAMPLE = MODE != S1_HIST_JBUF;
  static constexpr size_t kHistBytes = HIST ? (size_t)HistLayout<BMAX>::WORDS * sizeof(unsigned) : 0;
  using RG1 = Ring<FT, SAMPLE, HIST, !SAMPLE, 1, kSweep1Threads>;
  // as many ring slots (up to 4) as fit next to the histogram in 220 KiB
  static constexpr int NST_FIT = (int)((220 * 1024 - kHistBytes) / ((kSweep1Threads / 32) * (RG1::kSlot + 8)));
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;
  static_assert(NST >= 2, "ring needs two slots");
  using RG = Ring<FT, SAMPLE, HIST, !SAMPLE, NST, kSweep1Threads>;
  static constexpr size_t kSmem = kHistBytes + RG::kBytes;
};

template <typename MT, int BMAX, bool HIST, bool WRITEJ, bool WRITEG>
__device__ __forceinline__ void sweep1_half(const Half& H, unsigned* hist, const HistLane& hl, const Sweep1Args& a,
                                            bool sample) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < H.nv) {
      float d0, d1, d2, m[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) m[q] = tap_value<MT>(H.taps[j][q]);
      const float jv = sample ? interp8<WRITEG>(m, H.rr[j], d0, d1, d2) : H.x[j];
      if (HIST) hist_add<BMAX>(hist, hl, a.bf, a.bj, H.f[j], jv);
      if (WRITEJ) a.Jout[H.lin + 32u * j] = jv;
      if (WRITEG) {
        float* gp = a.Gout + 3ull * (H.lin + 32u * j);
        gp[0] = d0;
        gp[1] = d1;
        gp[2] = d2;
      }
    }
  }
}

template <typename FT, typename MT, int BMAX, int MODE, bool IA>
__global__ void __launch_bounds__(kSweep1Threads, 1) k_sweep1(const Sweep1Args a) {
  using C = S1Cfg<FT, BMAX, MODE>;
  constexpr bool HIST = C::HIST;
  constexpr bool SAMPLE = C::SAMPLE;
  constexpr bool WRITEG = (MODE == S1_HIST_WRITEJG) || (MODE == S1_WRITEJG);
  constexpr bool WRITEJ = (MODE == S1_WRITEJ) || (MODE == S1_HIST_WRITEJ) || WRITEG;
  constexpr int NST = C::NST;
  using L = HistLayout<BMAX>;
  using RG = typename C::RG;
  using WR = WarpRing<RG, NST>;
  extern __shared__ uint4 smem4[];
  unsigned* hist_sm = reinterpret_cast<unsigned*>(smem4);
  const Geom& g = a.g;
  HistLane hl;
  if (HIST) {
    hist_lane_init<BMAX>(hl);
    for (int i = threadIdx.x; i < L::WORDS / 4; i += kSweep1Threads) smem4[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  const float* X = a.Jin;
  WR wr;
  wr.init(reinterpret_cast<char*>(smem4) + C::kHistBytes, SAMPLE && a.u != nullptr);
  RingSched<WR, NST> rs{a.nIter, g.N / RG::kChunk, -1};
  const unsigned long long pol = policy_evict_first();
  rs.template prologue<FT>(wr, a.u, F, X, pol, a.stall_tx);
  LaneWalk w;
  Half A, B;
  unsigned k = 0;
  prepare<FT, MT, HIST, SAMPLE, !SAMPLE, SAMPLE, IA>(A, g, M, F, a.u, X, wr, rs, w, blockIdx.x, 0, 0, pol);
  int pending = 0;
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x, ++k) {
    prepare<FT, MT, HIST, SAMPLE, !SAMPLE, SAMPLE, IA>(B, g, M, F, a.u, X, wr, rs, w, it, k, 1, pol);
    sweep1_half<MT, BMAX, HIST, WRITEJ, WRITEG>(A, hist_sm, hl, a, SAMPLE);
    prepare<FT, MT, HIST, SAMPLE, !SAMPLE, SAMPLE, IA>(A, g, M, F, a.u, X, wr, rs, w, it + gridDim.x, k + 1, 0, pol);
    sweep1_half<MT, BMAX, HIST, WRITEJ, WRITEG>(B, hist_sm, hl, a, SAMPLE);
    if (HIST && ++pending == flush_every<BMAX, kSweep1Threads>()) {
      hist_flush<BMAX, kSweep1Threads>(hist_sm, a.ghist, a.B);
      pending = 0;
    }
  }
  rs.drain(wr);
  if (HIST) hist_flush<BMAX, kSweep1Threads>(hist_sm, a.ghist, a.B);
}

// ------------------------------------------------------------ MI finalize
// One CTA per histogram row a (BMAX CTAs; rows >= B are empty):
// P = H / (N 2^kHistFrac); marginals as row / column sums of the joint (equal
// to the separately defined marginals by partition of unity); the row's MI
// part sum_{b, P>0} P (ln P - ln P_F - ln P_J), added over rows in a fixed
// order by the finish kernel; and the row's entries of the gradient table of
// the scaled T = tscale (ln P - ln P_F - ln P_J) (0 where P = 0).  Every CTA
// recomputes the marginals (B^2 reads) so the logarithms, the costly part in
// fp64, are spread over BMAX SMs.
template <int BMAX>
__global__ void __launch_bounds__(256) k_mi_finalize(const FinalizeArgs a) {
  constexpr int TW = BMAX + 3;  // T columns -1 .. BMAX + 1
  __shared__ double P[BMAX * BMAX];
  __shared__ double lPF[BMAX], lPJ[BMAX];
  __shared__ double Ts[4][TW];  // unscaled T of rows a-1 .. a+2
  __shared__ double red[8];
  const int B = a.B, nb = B * B, tid = threadIdx.x, row = blockIdx.x;
  const double inv = 1.0 / (a.N * (double)kHistOne);
  for (int i = tid; i < nb; i += blockDim.x) P[i] = (double)a.ghist[i] * inv;
  __syncthreads();
  if (tid < B) {
    double s = 0.0;
    for (int c = 0; c < B; ++c) s += P[tid * B + c];
    lPF[tid] = s > 0.0 ? log(s) : 0.0;
  } else if (tid >= 128 && tid - 128 < B) {
    const int c = tid - 128;
    double s = 0.0;
    for (int r = 0; r < B; ++r) s += P[r * B + c];
    lPJ[c] = s > 0.0 ? log(s) : 0.0;
  }
  __syncthreads();
  for (int i = tid; i < 4 * TW; i += blockDim.x) {
    const int q = i / TW, c = i - q * TW - 1, ra = row - 1 + q;
    double t = 0.0;
    if (ra >= 0 && ra < B && c >= 0 && c < B) {
      const double p = P[ra * B + c];
      if (p > 0.0) t = log(p) - lPF[ra] - lPJ[c];
    }
    Ts[q][c + 1] = t;
  }
  __syncthreads();
  // this row's MI part
  double mi = 0.0;
  if (row < B && tid < B) mi = P[row * B + tid] * Ts[1][tid + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mi += __shfl_xor_sync(0xffffffffu, mi, o);
  if ((tid & 31) == 0) red[tid >> 5] = mi;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    a.scalars[row] = s;
  }
  const double ts = a.tscale;
  auto T = [&](int q, int c) -> double { return Ts[q][c + 1] * ts; };  // row a-1+q, column c
  // polynomial cell (row, fb): C[p][r] = sum_{ii,kk} T(row-1+ii, fb-1+kk) W[ii][p] D[kk][r]
  auto poly_cell = [&](int fb, float4* out) {
    const double W[4][4] = {{1.0 / 6, -0.5, 0.5, -1.0 / 6},
                            {2.0 / 3, 0.0, -1.0, 0.5},
                            {1.0 / 6, 0.5, 0.5, -0.5},
                            {0.0, 0.0, 0.0, 1.0 / 6}};
    // beta'(s) at s = (fb-1+k) - cJ as a polynomial in tJ:
    //   d0 = (1-t)^2/2, d1 = 2t - 1.5t^2, d2 = -1/2 - t + 1.5t^2, d3 = -t^2/2
    const double Dc[4][3] = {{0.5, -1.0, 0.5}, {0.0, 2.0, -1.5}, {-0.5, -1.0, 1.5}, {0.0, 0.0, -0.5}};
    double C[4][3] = {};
    for (int ii = 0; ii < 4; ++ii)
      for (int kk = 0; kk < 4; ++kk) {
        const double t = T(ii, fb - 1 + kk);
        if (t == 0.0) continue;
        for (int p = 0; p < 4; ++p)
          for (int r = 0; r < 3; ++r) C[p][r] += t * W[ii][p] * Dc[kk][r];
      }
    out[0] = make_float4((float)C[0][0], (float)C[0][1], (float)C[0][2], (float)C[1][0]);
    out[1] = make_float4((float)C[1][1], (float)C[1][2], (float)C[2][0], (float)C[2][1]);
    out[2] = make_float4((float)C[2][2], (float)C[3][0], (float)C[3][1], (float)C[3][2]);
  };
  if (tid < BMAX) {
    const int fb = tid, i = row * BMAX + fb;
    if constexpr (BMAX == 32) {
      poly_cell(fb, reinterpret_cast<float4*>(a.T) + 3 * i);
    } else {
      // rows of T packed as float2 pairs for the sweeps; polynomial cells for
      // the LNCC epilogue when requested
      reinterpret_cast<float2*>(a.T)[i] = make_float2((float)T(1, fb), (float)T(1, fb + 1));
      if (a.T2) poly_cell(fb, reinterpret_cast<float4*>(a.T2) + 3 * i);
    }
  }
}

// ------------------------------------------------------------------ sweep 2
// Per voxel g = dL/dJ (MI table or a given buffer), then either dJ (MI on a
// materialised J) or the sampler backward: du = K^T (g dJ/dq) and the affine
// partial sums, reduced per CTA in fp64.  Streams: u (sampling), F (MI), and
// g (given gradient) or J (MI on a given J).
template <typename FT, int BMAX, int MODE>
struct S2Cfg {
  static constexpr bool MI = MODE == S2_MI || MODE == S2_MI_JBUF || MODE == S2_MI_DJ;  // g from the MI table
  static constexpr bool MSE = MODE == S2_MSE;                                          // g = c (J - F)
  static constexpr bool GATHER = MODE == S2_MI || MODE == S2_GBUF || MSE;              // resample J and dJ/dq
  static constexpr bool VEC = GATHER || MODE == S2_GBUF_DJ || MODE == S2_MI_DJ;        // u or the stored dJ/dq
  static constexpr bool BWD = MODE != S2_MI_JBUF;                                      // du and affine partials
  static constexpr bool XS = MODE != S2_MI && !MSE;                                    // g or J (given / stored)
  static constexpr bool LF = MI || MSE;                                                // F streamed
  static constexpr int NACC = MSE ? 13 : 12;                                           // + sum (J - F)^2
  static constexpr size_t kTableBytes = MI ? (size_t)table_floats<BMAX>() * sizeof(float) : 0;
  static constexpr int NT = sweep2_threads(MODE);
  using RG1 = Ring<FT, VEC, LF, XS, 1, NT>;
  // as many ring slots (up to 4) as fit next to the table in 220 KiB
  static constexpr int NST_FIT = (int)((220 * 1024 - kTableBytes - (NT / 32) * 96) / ((NT / 32) * (RG1::kSlot + 8)));
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;
  static_assert(NST >= 2, "ring needs two slots");
  using RG = Ring<FT, VEC, LF, XS, NST, NT>;
  static constexpr size_t kSmem = kTableBytes + RG::kBytes;
};

template <typename MT, int BMAX, bool MI, bool GATHER, bool BWD, bool MSE = false>
__device__ __forceinline__ void sweep2_half(const Half& H, const float* tsm, const Sweep2Args& a,
                                            float acc[MSE ? 13 : 12]) {
  const Geom& g = a.g;
  if constexpr (!BWD) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (j < H.nv) a.dJ[H.lin + 32u * j] = mi_grad<BMAX>(tsm, a.bf, a.bj, H.f[j], H.x[j]);
  } else {
    float e[2][3];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      e[j][0] = e[j][1] = e[j][2] = 0.0f;
      if (j >= H.nv) continue;
      float gq0, gq1, gq2, gv;
      if (GATHER) {
        float m[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) m[q] = tap_value<MT>(H.taps[j][q]);
        const float jv = interp8<true>(m, H.rr[j], gq0, gq1, gq2);
        if constexpr (MSE) {
          const float d = jv - H.f[j];
          gv = a.mse_c * d;
          acc[12] = fmaf(d, d, acc[12]);  // this thread's sum (J - F)^2
        } else {
          gv = MI ? mi_grad<BMAX>(tsm, a.bf, a.bj, H.f[j], jv) : H.x[j];
        }
      } else {
        // the stored slope of J, and g given or from the MI table at the stored J
        gq0 = H.rr[j][0];
        gq1 = H.rr[j][1];
        gq2 = H.rr[j][2];
        gv = MI ? mi_grad<BMAX>(tsm, a.bf, a.bj, H.f[j], H.x[j]) : H.x[j];
      }
      e[j][0] = gv * gq0;
      e[j][1] = gv * gq1;
      e[j][2] = gv * gq2;
      if (a.du) {
        float o0, o1, o2;
        if (g.k_diag) {
          o0 = g.K[0] * e[j][0];
          o1 = g.K[4] * e[j][1];
          o2 = g.K[8] * e[j][2];
        } else {
          o0 = fmaf(g.K[0], e[j][0], fmaf(g.K[3], e[j][1], g.K[6] * e[j][2]));
          o1 = fmaf(g.K[1], e[j][0], fmaf(g.K[4], e[j][1], g.K[7] * e[j][2]));
          o2 = fmaf(g.K[2], e[j][0], fmaf(g.K[5], e[j][1], g.K[8] * e[j][2]));
        }
        float* dp = a.du + 3ull * (H.lin + 32u * j);
        dp[0] = o0;
        dp[1] = o1;
        dp[2] = o2;
      }
      const float cx = (float)H.ix[j] - g.ctr[0];
#pragma unroll
      for (int r = 0; r < 3; ++r) acc[kPM + 3 * r] = fmaf(e[j][r], cx, acc[kPM + 3 * r]);
    }
    // the two voxels of a half share (y, z) unless a row ends between them:
    // their y and z moments then take one product per half
    const float s[3] = {e[0][0] + e[1][0], e[0][1] + e[1][1], e[0][2] + e[1][2]};
#pragma unroll
    for (int r = 0; r < 3; ++r) acc[kPS + r] += s[r];
    if (H.nv == 2 && (H.iy[0] != H.iy[1] || H.iz[0] != H.iz[1])) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float cy = (float)H.iy[j] - g.ctr[1], cz = (float)H.iz[j] - g.ctr[2];
#pragma unroll
        for (int r = 0; r < 3; ++r) {
          acc[kPM + 3 * r + 1] = fmaf(e[j][r], cy, acc[kPM + 3 * r + 1]);
          acc[kPM + 3 * r + 2] = fmaf(e[j][r], cz, acc[kPM + 3 * r + 2]);
        }
      }
    } else {
      const float cy = (float)H.iy[0] - g.ctr[1], cz = (float)H.iz[0] - g.ctr[2];
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        acc[kPM + 3 * r + 1] = fmaf(s[r], cy, acc[kPM + 3 * r + 1]);
        acc[kPM + 3 * r + 2] = fmaf(s[r], cz, acc[kPM + 3 * r + 2]);
      }
    }
  }
}

template <typename FT, typename MT, int BMAX, int MODE, bool IA>
__global__ void __launch_bounds__(sweep2_threads(MODE), 1) k_sweep2(const Sweep2Args a) {
  using C = S2Cfg<FT, BMAX, MODE>;
  constexpr bool MI = C::MI, GATHER = C::GATHER, VEC = C::VEC, BWD = C::BWD, XS = C::XS, MSE = C::MSE;
  constexpr bool LF = C::LF;
  constexpr int NST = C::NST, NACC = C::NACC;
  using RG = typename C::RG;
  using WR = WarpRing<RG, NST>;
  extern __shared__ float4 tsm4[];
  float* tsm = reinterpret_cast<float*>(tsm4);
  constexpr int NT = C::NT;
  __shared__ double wsum[NT / 32][NACC];
  const Geom& g = a.g;
  if (MI) {
    constexpr int n4 = table_floats<BMAX>() / 4;
    const float4* src = reinterpret_cast<const float4*>(a.T);
    for (int i = threadIdx.x; i < n4; i += NT) tsm4[i] = __ldg(src + i);
    __syncthreads();
  }
  const FT* __restrict__ F = static_cast<const FT*>(a.F);
  const MT* __restrict__ M = static_cast<const MT*>(a.M);
  const float* X = (MODE == S2_MI_JBUF || MODE == S2_MI_DJ) ? a.Jin : a.gbuf;
  const float* U = GATHER ? a.u : a.dJdq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (BWD && lane == 0)
#pragma unroll
    for (int q = 0; q < NACC; ++q) wsum[warp][q] = 0.0;
  float acc[NACC];
#pragma unroll
  for (int q = 0; q < NACC; ++q) acc[q] = 0.0f;
  WR wr;
  wr.init(reinterpret_cast<char*>(tsm4) + C::kTableBytes, VEC && U != nullptr);
  RingSched<WR, NST> rs{a.nIter, g.N / RG::kChunk, -1};
  const unsigned long long pol = policy_evict_first();
  rs.template prologue<FT>(wr, U, F, X, pol);
  LaneWalk w;
  Half A, B;
  unsigned k = 0;
  if constexpr (GATHER) prepare<FT, MT, LF, VEC, XS, GATHER, IA>(A, g, M, F, U, X, wr, rs, w, blockIdx.x, 0, 0, pol);
  int pending = 0;
  for (unsigned it = blockIdx.x; it < a.nIter; it += gridDim.x, ++k) {
    if constexpr (GATHER) {
      // gathers of the next half are in flight while the current one computes
      prepare<FT, MT, LF, VEC, XS, GATHER, IA>(B, g, M, F, U, X, wr, rs, w, it, k, 1, pol);
      sweep2_half<MT, BMAX, MI, GATHER, BWD, MSE>(A, tsm, a, acc);
      prepare<FT, MT, LF, VEC, XS, GATHER, IA>(A, g, M, F, U, X, wr, rs, w, it + gridDim.x, k + 1, 0, pol);
      sweep2_half<MT, BMAX, MI, GATHER, BWD, MSE>(B, tsm, a, acc);
    } else {
      prepare_chunk<FT, MI, VEC, XS>(A, B, g, F, U, X, wr, rs, it, k, pol);
      sweep2_half<MT, BMAX, MI, GATHER, BWD>(A, tsm, a, acc);
      sweep2_half<MT, BMAX, MI, GATHER, BWD>(B, tsm, a, acc);
    }
    if (BWD && ++pending == kFoldEvery) {
#pragma unroll
      for (int q = 0; q < NACC; ++q) {
        const float s = warp_sum(acc[q]);
        if (lane == 0) wsum[warp][q] += (double)s;
        acc[q] = 0.0f;
      }
      pending = 0;
    }
  }
  rs.drain(wr);
  if (BWD) {
#pragma unroll
    for (int q = 0; q < NACC; ++q) {
      const float s = warp_sum(acc[q]);
      if (lane == 0) wsum[warp][q] += (double)s;
    }
    __syncthreads();
    if (threadIdx.x < kPartialStride) {
      // acc[12] (MSE) goes to record slot kPSE; slot kPCC stays 0
      const int q = threadIdx.x < 12 ? (int)threadIdx.x : (MSE && threadIdx.x == kPSE ? 12 : -1);
      double s = 0.0;
      if (q >= 0)
        for (int w2 = 0; w2 < NT / 32; ++w2) s += wsum[w2][q];
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
    if (a.loss && g_ffdp_device_error) {
      for (int i = 0; i < a.nloss; ++i) a.loss[i] = __int_as_float(0x7fc00000);  // a ring wait gave up: NaN
    } else if (a.loss) {
      double mi = 0.0;
      if (a.has_mi)
        for (int r = 0; r < a.mi_rows; ++r) mi += a.scalars[r];  // fixed order
      const double lncc = a.has_lncc ? sm[kPCC][16] / a.N : 0.0;
      const double mse = a.has_mse ? sm[kPSE][16] / a.N : 0.0;
      if (a.has_mse) {
        if (a.nloss == 2) {
          a.loss[0] = (float)(a.w_mse * mse);
          a.loss[1] = (float)mse;
        } else {
          a.loss[0] = (float)mse;
        }
      } else if (a.nloss == 3) {
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
static cudaError_t run_sweep1(const Sweep1Args& a, int grid, cudaStream_t s, int* occ) {
  constexpr bool SAMPLE = S1Cfg<FT, BMAX, MODE>::SAMPLE;
  auto k = (SAMPLE && a.g.ia) ? k_sweep1<FT, MT, BMAX, MODE, SAMPLE> : k_sweep1<FT, MT, BMAX, MODE, false>;
  const size_t smem = S1Cfg<FT, BMAX, MODE>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, kSweep1Threads, smem);
  note_launch_begin("k_sweep1", s);
  k<<<grid, kSweep1Threads, smem, s>>>(a);
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
        case S1_HIST_WRITEJG: e = run_sweep1<FT, MT, 32, S1_HIST_WRITEJG>(a, grid, s, occ); break;
        case S1_WRITEJG: e = run_sweep1<float, MT, 32, S1_WRITEJG>(a, grid, s, occ); break;
      }
    } else {
      switch (mode) {
        case S1_HIST: e = run_sweep1<FT, MT, 64, S1_HIST>(a, grid, s, occ); break;
        case S1_HIST_WRITEJ: e = run_sweep1<FT, MT, 64, S1_HIST_WRITEJ>(a, grid, s, occ); break;
        case S1_WRITEJ: e = run_sweep1<float, MT, 32, S1_WRITEJ>(a, grid, s, occ); break;
        case S1_HIST_JBUF: e = run_sweep1<FT, float, 64, S1_HIST_JBUF>(a, grid, s, occ); break;
        case S1_HIST_WRITEJG: e = run_sweep1<FT, MT, 64, S1_HIST_WRITEJG>(a, grid, s, occ); break;
        case S1_WRITEJG: e = run_sweep1<float, MT, 32, S1_WRITEJG>(a, grid, s, occ); break;
      }
    }
  }));
  return e;
}

cudaError_t launch_sweep1(int mode, int ft, int mt, int bmax, const Sweep1Args& a, int grid, cudaStream_t s) {
  return dispatch_sweep1(mode, ft, mt, bmax, a, grid, s, nullptr);
}

int sweep1_ctas_per_sm(int mode, int ft, int mt, int bmax) {
  static OccCache<kSweep1Modes * 8> cache;
  return cache.get(((mode * 2 + ft) * 2 + mt) * 2 + (bmax == 64), [&] {
    int occ = 0;
    Sweep1Args dummy{};
    return dispatch_sweep1(mode, ft, mt, bmax, dummy, 0, 0, &occ) == cudaSuccess ? occ : 1;
  });
}

template <typename FT, typename MT, int BMAX, int MODE>
static cudaError_t run_sweep2(const Sweep2Args& a, int grid, cudaStream_t s, int* occ) {
  constexpr bool GATHER = S2Cfg<FT, BMAX, MODE>::GATHER;
  auto k = (GATHER && a.g.ia) ? k_sweep2<FT, MT, BMAX, MODE, GATHER> : k_sweep2<FT, MT, BMAX, MODE, false>;
  const size_t smem = S2Cfg<FT, BMAX, MODE>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int nt = S2Cfg<FT, BMAX, MODE>::NT;
  if (occ) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, nt, smem);
  note_launch_begin("k_sweep2", s);
  k<<<grid, nt, smem, s>>>(a);
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
        case S2_GBUF_DJ: e = run_sweep2<float, float, 32, S2_GBUF_DJ>(a, grid, s, occ); break;
        case S2_MI_DJ: e = run_sweep2<FT, float, 32, S2_MI_DJ>(a, grid, s, occ); break;
        case S2_MSE: e = run_sweep2<FT, MT, 32, S2_MSE>(a, grid, s, occ); break;
      }
    } else {
      switch (mode) {
        case S2_MI: e = run_sweep2<FT, MT, 64, S2_MI>(a, grid, s, occ); break;
        case S2_GBUF: e = run_sweep2<float, MT, 32, S2_GBUF>(a, grid, s, occ); break;
        case S2_MI_JBUF: e = run_sweep2<FT, float, 64, S2_MI_JBUF>(a, grid, s, occ); break;
        case S2_GBUF_DJ: e = run_sweep2<float, float, 32, S2_GBUF_DJ>(a, grid, s, occ); break;
        case S2_MI_DJ: e = run_sweep2<FT, float, 64, S2_MI_DJ>(a, grid, s, occ); break;
        case S2_MSE: e = run_sweep2<FT, MT, 32, S2_MSE>(a, grid, s, occ); break;
      }
    }
  }));
  return e;
}

cudaError_t launch_sweep2(int mode, int ft, int mt, int bmax, const Sweep2Args& a, int grid, cudaStream_t s) {
  return dispatch_sweep2(mode, ft, mt, bmax, a, grid, s, nullptr);
}

int sweep2_ctas_per_sm(int mode, int ft, int mt, int bmax) {
  static OccCache<kSweep2Modes * 8> cache;
  return cache.get(((mode * 2 + ft) * 2 + mt) * 2 + (bmax == 64), [&] {
    int occ = 0;
    Sweep2Args dummy{};
    return dispatch_sweep2(mode, ft, mt, bmax, dummy, 0, 0, &occ) == cudaSuccess ? occ : 1;
  });
}

cudaError_t launch_finalize(int bmax, const FinalizeArgs& a, cudaStream_t s) {
  note_launch_begin("k_mi_finalize", s);
  if (bmax == 32)
    k_mi_finalize<32><<<32, 256, 0, s>>>(a);
  else
    k_mi_finalize<64><<<64, 256, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t launch_finish(const FinishArgs& a, cudaStream_t s) {
  note_launch_begin("k_finish", s);
  k_finish<<<1, 256, 0, s>>>(a);
  note_launch_end(s);
  return cudaGetLastError();
}

cudaError_t take_device_error(unsigned* v) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_ffdp_device_error, sizeof(unsigned));
  if (e == cudaSuccess && *v) {
    const unsigned zero = 0u;
    e = cudaMemcpyToSymbol(g_ffdp_device_error, &zero, sizeof(unsigned));
  }
  return e;
}

size_t mi_table_bytes(int bmax) { return (size_t)(bmax == 32 ? table_floats<32>() : table_floats<64>()) * sizeof(float); }

}  // namespace ffdp
