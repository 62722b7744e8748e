// ffdp_api.cu -- the C ABI of libffdp (declared in include/ffdp.h): argument
// validation, transform pre-computation, workspace layout and the launch
// pipeline of each entry point.
//
// Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
// Registration", Key designs items 1 (fused_grid_sampler(I; A, t, [u], S,
// x_bounds)) and 2 (implicit-Parzen MI, fused LNCC); "Background" for the
// objective L = C(F, M o phi), phi(x) = Ax + t + u(x).
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/ffdp.h"
#include "ffdp_internal.h"
#include "ffdp_reg.h"

using namespace ffdp;

// ------------------------------------------------------------ error detail
static thread_local char g_err[512] = "";

static ffdp_status fail(ffdp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

static ffdp_status cuda_fail(cudaError_t e, const char* where) {
  return fail(FFDP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

extern "C" const char* ffdp_last_error(void) { return g_err; }

extern "C" const char* ffdp_status_string(ffdp_status s) {
  switch (s) {
    case FFDP_OK: return "FFDP_OK";
    case FFDP_ERR_INVALID_ARGUMENT: return "FFDP_ERR_INVALID_ARGUMENT";
    case FFDP_ERR_UNSUPPORTED: return "FFDP_ERR_UNSUPPORTED";
    case FFDP_ERR_WORKSPACE: return "FFDP_ERR_WORKSPACE";
    case FFDP_ERR_CUDA: return "FFDP_ERR_CUDA";
    case FFDP_ERR_INTERNAL: return "FFDP_ERR_INTERNAL";
  }
  return "FFDP_ERR_UNKNOWN";
}

// -------------------------------------------------- launch accounting
namespace {
std::atomic<unsigned long long> g_launches{0};
struct TimingRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_tmu;
std::vector<cudaEvent_t> g_events;  // pool, 2 per record
std::vector<TimingRec> g_recs;
int g_cap = 0;
thread_local int g_open = -1;  // record index opened by note_launch_begin
}  // namespace

void ffdp::note_launch_begin(const char* name, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  g_open = -1;
  if (g_cap == 0) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  const int i = (int)g_recs.size();
  if (i >= g_cap) return;
  TimingRec r{name, g_events[2 * i], g_events[2 * i + 1]};
  cudaEventRecord(r.a, s);
  g_recs.push_back(r);
  g_open = i;
}

void ffdp::note_launch_end(cudaStream_t s) {
  if (g_open < 0) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  cudaEventRecord(g_recs[g_open].b, s);
  g_open = -1;
}

extern "C" uint64_t ffdp_launch_count(void) { return g_launches.load(); }

namespace {
std::atomic<unsigned> g_test_stall{0};
}

unsigned ffdp::take_test_stall() { return g_test_stall.exchange(0u); }

extern "C" ffdp_status ffdp_test_ring_stall(int on) {
  g_test_stall.store(on ? 16u : 0u);
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_device_error(int* flag) {
  if (!flag) return fail(FFDP_ERR_INVALID_ARGUMENT, "flag is NULL");
  unsigned v = 0;
  const cudaError_t e = ffdp::take_device_error(&v);
  if (e != cudaSuccess) return cuda_fail(e, "device error word");
  *flag = v ? 1 : 0;
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_timing_enable(int capacity) {
  std::lock_guard<std::mutex> lk(g_tmu);
  g_recs.clear();
  if (capacity < 0) return fail(FFDP_ERR_INVALID_ARGUMENT, "timing capacity < 0");
  const size_t need = 2 * (size_t)capacity;
  while (g_events.size() < need) {
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventCreate");
    g_events.push_back(e);
  }
  g_cap = capacity;
  return FFDP_OK;
}

extern "C" int ffdp_timing_read(char* names, int* counts, double* ms, int max) {
  std::lock_guard<std::mutex> lk(g_tmu);
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> tot;
  for (const TimingRec& r : g_recs) {
    cudaEventSynchronize(r.b);
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) t = 0.0f;
    size_t k = 0;
    while (k < keys.size() && keys[k] != r.name) ++k;
    if (k == keys.size()) {
      keys.push_back(r.name);
      cnt.push_back(0);
      tot.push_back(0.0);
    }
    cnt[k] += 1;
    tot[k] += t;
  }
  for (size_t k = 0; k < keys.size() && (int)k < max; ++k) {
    if (names) {
      std::strncpy(names + 64 * k, keys[k].c_str(), 63);
      names[64 * k + 63] = '\0';
    }
    if (counts) counts[k] = cnt[k];
    if (ms) ms[k] = tot[k];
  }
  return (int)keys.size();
}

// --------------------------------------------------------- helpers
namespace {

constexpr int64_t kMaxDim = 1 << 20;
constexpr uint64_t kMaxVoxels = (1ull << 32) - (1ull << 16);

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

ffdp_status check_dims(ffdp_dims d, const char* what) {
  if (d.d < 2 || d.h < 2 || d.w < 2)
    return fail(FFDP_ERR_INVALID_ARGUMENT, "%s dims must be >= 2 (got %lld x %lld x %lld)", what,
                (long long)d.d, (long long)d.h, (long long)d.w);
  if (d.d > kMaxDim || d.h > kMaxDim || d.w > kMaxDim)
    return fail(FFDP_ERR_UNSUPPORTED, "%s dims above 2^20", what);
  if ((uint64_t)d.d * (uint64_t)d.h * (uint64_t)d.w > kMaxVoxels)
    return fail(FFDP_ERR_UNSUPPORTED, "%s has more than 2^32 - 2^16 voxels", what);
  return FFDP_OK;
}

ffdp_status check_dtype(ffdp_dtype t, const char* what) {
  if (t != FFDP_F32 && t != FFDP_F16) return fail(FFDP_ERR_INVALID_ARGUMENT, "%s dtype must be F32 or F16", what);
  return FFDP_OK;
}

uint64_t nvox(ffdp_dims d) { return (uint64_t)d.d * (uint64_t)d.h * (uint64_t)d.w; }

// magic numbers for fast_div (round-up method): s = ceil(log2 d),
// m = floor(2^32 (2^s - d) / d) + 1, q = (umulhi(n, m) + n) >> s.
void fast_div_magic(uint32_t d, unsigned& m, int& s) {
  int l = 0;
  while ((1ull << l) < d) ++l;
  const unsigned __int128 num = ((unsigned __int128)1 << 32) * (((unsigned __int128)1 << l) - d);
  m = (unsigned)(num / d + 1);
  s = l;
}

ffdp_status make_geom(ffdp_dims f, ffdp_dims m, const ffdp_transform* T, Geom& g) {
  const double nf[3] = {(double)f.w, (double)f.h, (double)f.d};
  const double nm[3] = {(double)m.w, (double)m.h, (double)m.d};
  for (int k = 0; k < 9; ++k)
    if (!std::isfinite(T->A[k]) || !std::isfinite(T->S[k]))
      return fail(FFDP_ERR_INVALID_ARGUMENT, "non-finite A or S");
  for (int k = 0; k < 3; ++k)
    if (!std::isfinite(T->t[k]) || !std::isfinite(T->xmin[k]) || !std::isfinite(T->xmax[k]))
      return fail(FFDP_ERR_INVALID_ARGUMENT, "non-finite t or x_bounds");
  double dx[3], hM[3];
  for (int c = 0; c < 3; ++c) {
    dx[c] = ((double)T->xmax[c] - (double)T->xmin[c]) / (nf[c] - 1.0);
    hM[c] = (nm[c] - 1.0) / 2.0;
  }
  const double two32 = 4294967296.0;
  if ((uint64_t)m.d * (uint64_t)m.h * (uint64_t)m.w >= (1ull << 31))
    return fail(FFDP_ERR_UNSUPPORTED, "moving image has 2^31 or more voxels");
  for (int r = 0; r < 3; ++r) {
    double g0 = (double)T->t[r] + 1.0;
    double reach = 0.0;  // largest |G i| over the fixed grid
    for (int c = 0; c < 3; ++c) {
      const double G = hM[r] * (double)T->A[r * 3 + c] * dx[c];
      reach += std::fabs(G) * (nf[c] - 1.0);
      g.Gq[r * 3 + c] = (long long)llround(G * two32);
      g0 += (double)T->A[r * 3 + c] * (double)T->xmin[c];
      g.K[r * 3 + c] = (float)(hM[r] * (double)T->S[r * 3 + c]);
    }
    g0 *= hM[r];
    // keeps the integer part of every anchor below 2^25 voxels
    if (reach + std::fabs(g0) > 16777216.0) return fail(FFDP_ERR_UNSUPPORTED, "affine maps the grid beyond 2^24 voxels");
    g.g0q[r] = (long long)llround(g0 * two32);
    g.Gx[r] = (float)(hM[r] * (double)T->A[r * 3 + 0] * dx[0]);
    g.hM[r] = (float)hM[r];
    g.ctr[r] = (float)((nf[r] - 1.0) / 2.0);
  }
  g.a_diag = (g.Gq[1] == 0 && g.Gq[2] == 0 && g.Gq[3] == 0 && g.Gq[5] == 0 && g.Gq[6] == 0 && g.Gq[7] == 0) ? 1 : 0;
  g.k_diag = (T->S[1] == 0.f && T->S[2] == 0.f && T->S[3] == 0.f && T->S[5] == 0.f && T->S[6] == 0.f &&
              T->S[7] == 0.f)
                 ? 1
                 : 0;
  const long long one = 1ll << 32;
  g.ia = (g.a_diag && g.Gq[0] == one && g.Gq[4] == one && g.Gq[8] == one && (g.g0q[0] & (one - 1)) == 0 &&
          (g.g0q[1] & (one - 1)) == 0 && (g.g0q[2] & (one - 1)) == 0)
             ? 1
             : 0;
  for (int c = 0; c < 3; ++c) g.io[c] = g.ia ? (int)(g.g0q[c] >> 32) : 0;
  g.fW = (int)f.w;
  g.fH = (int)f.h;
  g.fD = (int)f.d;
  g.mW = (int)m.w;
  g.mH = (int)m.h;
  g.mD = (int)m.d;
  g.mHW = (long long)m.w * m.h;
  g.N = (unsigned)nvox(f);
  fast_div_magic((uint32_t)f.w, g.divW_m, g.divW_s);
  fast_div_magic((uint32_t)(f.w * f.h), g.divHW_m, g.divHW_s);
  return FFDP_OK;
}

// Extents only (for ops without a sampler).
void make_grid_only(ffdp_dims f, Geom& g) {
  std::memset(&g, 0, sizeof(g));
  g.fW = (int)f.w;
  g.fH = (int)f.h;
  g.fD = (int)f.d;
  g.N = (unsigned)nvox(f);
  fast_div_magic((uint32_t)f.w, g.divW_m, g.divW_s);
  fast_div_magic((uint32_t)(f.w * f.h), g.divHW_m, g.divHW_s);
}

ffdp_status check_mi(const ffdp_mi_params* p) {
  if (!p) return fail(FFDP_ERR_INVALID_ARGUMENT, "null MI params");
  if (p->bins < 8 || p->bins > 64) return fail(FFDP_ERR_INVALID_ARGUMENT, "bins must be in [8, 64]");
  if (!std::isfinite(p->f_lo) || !std::isfinite(p->f_hi) || !(p->f_hi > p->f_lo))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "fixed intensity range needs finite f_lo < f_hi");
  if (!std::isfinite(p->m_lo) || !std::isfinite(p->m_hi) || !(p->m_hi > p->m_lo))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "moving intensity range needs finite m_lo < m_hi");
  return FFDP_OK;
}

ffdp_status check_lncc(const ffdp_lncc_params* p) {
  if (!p) return fail(FFDP_ERR_INVALID_ARGUMENT, "null LNCC params");
  if (p->window < 3 || (p->window & 1) == 0) return fail(FFDP_ERR_INVALID_ARGUMENT, "window must be odd and >= 3");
  if (!std::isfinite(p->eps) || p->eps < 0.0f) return fail(FFDP_ERR_INVALID_ARGUMENT, "eps must be finite and >= 0");
  return FFDP_OK;
}

BinMap bin_map(float lo, float hi, int B) {
  BinMap m;
  const double sc = (double)(B - 5) / ((double)hi - (double)lo);
  m.lo = lo;
  m.hi = hi;
  m.sc = (float)sc;
  m.off = (float)(2.0 - (double)lo * sc);
  return m;
}

int bmax_of(int bins) { return bins <= 32 ? 32 : 64; }

// Workspace layout (byte offsets, 256-aligned).
struct Ws {
  size_t hist, table, table2, scalars, partials, J, DG, WA, WB, GS, total;
};

// The LNCC window runs through the wide-window passes (two [5][N] buffers).
bool lncc_wide(int window) { return window > kLnccTiledMaxWindow; }

// The tiled LNCC runs as the forward / backward kernel pair, with the g-terms
// ([3][N]) in the workspace.
bool lncc_split(int window) { return kLnccSplit && !kLnccRecompute && !lncc_wide(window); }

// Window radius of the wide-window passes: a radius at or beyond the largest
// grid extent sums the same (clipped) terms, so it is capped there; the
// divisor stays the true window^3.
int wide_radius(int window, const Geom& g) {
  const int R = (window - 1) / 2;
  const int e = std::max(g.fW, std::max(g.fH, g.fD));
  return R < e ? R : e;
}

size_t al(size_t x) { return (x + 255) & ~(size_t)255; }

// True when the LNCC objective samples J on chip instead of storing it (the
// halo-recompute build, window radius <= 3).
bool lncc_recompute(int window) { return kLnccRecompute && window <= 7; }

// ln: LNCC on; store: J and dJ/dq per voxel.
Ws ws_layout(bool mi, int bmax, size_t max_parts, bool ln, bool store, uint64_t N, bool wide = false,
             bool split = false) {
  const bool needJ = store;
  Ws w;
  size_t o = 0;
  w.hist = o;
  if (mi) o = al(o + (size_t)bmax * bmax * sizeof(unsigned long long));
  w.table = o;
  if (mi) o = al(o + mi_table_bytes(bmax));
  w.table2 = o;
  // the LNCC epilogue reads polynomial cells: the main table for 32 bins, this one for 64
  if (mi && ln && bmax == 64) o = al(o + (size_t)bmax * bmax * 12 * sizeof(float));
  w.scalars = o;
  o = al(o + 64 * sizeof(double));  // MI part per histogram row
  w.partials = o;  // one record per CTA of the last kernel of the path
  o = al(o + max_parts * kPartialStride * sizeof(double));
  w.J = o;
  if (needJ) o = al(o + (size_t)N * sizeof(float));
  w.DG = o;  // dJ/dq, [N][3]
  if (needJ) o = al(o + (size_t)N * 3 * sizeof(float));
  w.WA = o;  // wide-window LNCC: window sums, then g-terms, [5][N] each
  if (wide) o = al(o + (size_t)N * 5 * sizeof(float));
  w.WB = o;
  if (wide) o = al(o + (size_t)N * 5 * sizeof(float));
  w.GS = o;  // split LNCC: the g-terms, [3][N]
  if (split) o = al(o + (size_t)N * 3 * sizeof(float));
  w.total = o;
  return w;
}

size_t max_parts() { return (size_t)(sm_count() > 0 ? sm_count() : 1) * kMaxCtasPerSm; }

ffdp_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return FFDP_OK;
  if (!ws) return fail(FFDP_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
  if (ws_bytes < need) return fail(FFDP_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need, ws_bytes);
  if (!aligned16(ws)) return fail(FFDP_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  return FFDP_OK;
}

int persistent_grid(unsigned nIter, int per_sm) {
  long long g = (long long)sm_count() * per_sm;
  if (g < 1) g = 1;
  if ((long long)nIter < g) g = nIter;
  return (int)(g < 1 ? 1 : g);
}

// CTA iterations of the histogram / forward sweep and of the gradient sweep
unsigned n_iter1(uint64_t N) {
  return (unsigned)((N + (uint64_t)(kSweep1Threads * kVPT) - 1) / (kSweep1Threads * kVPT));
}
unsigned n_iter2(uint64_t N, int mode) {
  const uint64_t per = (uint64_t)sweep2_threads(mode) * kVPT;
  return (unsigned)((N + per - 1) / per);
}

#define FFDP_TRY(x)                    \
  do {                                 \
    ffdp_status _st = (x);             \
    if (_st != FFDP_OK) return _st;    \
  } while (0)

#define FFDP_CUDA(x, where)                          \
  do {                                               \
    cudaError_t _e = (x);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, where); \
  } while (0)

// LNCC tiling for a fixed grid: one resident CTA per slot, each taking an
// equal run of the (column, plane) sequence over (32 x TY) columns, at least
// 32 planes per CTA.
void lncc_tiling(ffdp_dims f, int R, LnccArgs& a, int per_sm, int& grid) {
  const int TY = lncc_ty(R);
  a.tilesX = (int)((f.w + kLnccTX - 1) / kLnccTX);
  a.tilesY = (int)((f.h + TY - 1) / TY);
  const long long total = (long long)a.tilesX * a.tilesY * (long long)f.d;
  const long long slots = (long long)sm_count() * per_sm;
  long long n = (total + 31) / 32;
  if (n > slots) n = slots;
  if (n < 1) n = 1;
  a.per = (total + n - 1) / n;
  grid = (int)((total + a.per - 1) / a.per);
}

}  // namespace

// ---------------------------------------------------------------- ABI
extern "C" size_t ffdp_workspace_bytes(int op, ffdp_dims fixed, const void* params) {
  if (check_dims(fixed, "fixed") != FFDP_OK) return 0;
  const uint64_t N = nvox(fixed);
  switch (op) {
    case FFDP_OP_GRID_SAMPLE_BWD:
      return ws_layout(false, 32, max_parts(), false, false, N).total;
    case FFDP_OP_MI: {
      const ffdp_mi_params* p = static_cast<const ffdp_mi_params*>(params);
      if (check_mi(p) != FFDP_OK) return 0;
      return ws_layout(true, bmax_of(p->bins), max_parts(), false, false, N).total;
    }
    case FFDP_OP_LNCC: {
      const ffdp_lncc_params* p = static_cast<const ffdp_lncc_params*>(params);
      if (check_lncc(p) != FFDP_OK) return 0;
      return ws_layout(false, 32, max_parts(), false, false, N, lncc_wide(p->window), lncc_split(p->window)).total;
    }
    case FFDP_OP_OBJECTIVE:
    case FFDP_OP_OBJECTIVE_STORED: {
      const ffdp_objective_params* p = static_cast<const ffdp_objective_params*>(params);
      if (!p) return 0;
      const bool mi = p->w_mi != 0.0f, ln = p->w_lncc != 0.0f;
      if (mi && check_mi(&p->mi) != FFDP_OK) return 0;
      if (ln && check_lncc(&p->lncc) != FFDP_OK) return 0;
      const bool store_slope = op == FFDP_OP_OBJECTIVE_STORED;
      return ws_layout(mi, mi ? bmax_of(p->mi.bins) : 32, max_parts(), ln,
                       (ln && !lncc_recompute(p->lncc.window)) || (mi && !ln && store_slope), N,
                       ln && lncc_wide(p->lncc.window), ln && lncc_split(p->lncc.window)).total;
    }
    case FFDP_OP_SAMPLE_CHANNELS_BWD:
    case FFDP_OP_MSE:
    case FFDP_OP_OBJECTIVE_MSE:
    case FFDP_OP_SOBOLEV:
      return ws_layout(false, 32, max_parts(), false, false, N).total;
  }
  return 0;
}

extern "C" ffdp_status ffdp_grid_sample_fwd(const void* M, ffdp_dtype mt, ffdp_dims mdims, ffdp_dims out_dims,
                                            const float* u, const ffdp_transform* T, float* J_out,
                                            void* stream) {
  g_err[0] = '\0';
  if (!M || !T || !J_out) return fail(FFDP_ERR_INVALID_ARGUMENT, "null M, T or J_out");
  FFDP_TRY(check_dtype(mt, "M"));
  FFDP_TRY(check_dims(mdims, "moving"));
  FFDP_TRY(check_dims(out_dims, "output"));
  if (!aligned16(J_out) || (u && !aligned16(u))) return fail(FFDP_ERR_INVALID_ARGUMENT, "J_out and u must be 16-byte aligned");
  Sweep1Args a{};
  FFDP_TRY(make_geom(out_dims, mdims, T, a.g));
  a.M = M;
  a.u = u;
  a.Jout = J_out;
  a.nIter = n_iter1(a.g.N);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = persistent_grid(a.nIter, sweep1_ctas_per_sm(S1_WRITEJ, 0, mt, 32));
  FFDP_CUDA(launch_sweep1(S1_WRITEJ, 0, mt, 32, a, grid, s), "grid_sample_fwd launch");
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_grid_sample_bwd(const void* M, ffdp_dtype mt, ffdp_dims mdims, ffdp_dims out_dims,
                                            const float* u, const ffdp_transform* T, const float* gJ,
                                            float* du, float* dA, float* dt, void* ws, size_t ws_bytes,
                                            void* stream) {
  g_err[0] = '\0';
  if (!M || !T || !gJ) return fail(FFDP_ERR_INVALID_ARGUMENT, "null M, T or gJ");
  FFDP_TRY(check_dtype(mt, "M"));
  FFDP_TRY(check_dims(mdims, "moving"));
  FFDP_TRY(check_dims(out_dims, "output"));
  if ((u && !aligned16(u)) || !aligned16(gJ) || (du && !aligned16(du)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "u, gJ and du must be 16-byte aligned");
  const Ws w = ws_layout(false, 32, max_parts(), false, false, nvox(out_dims));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  Sweep2Args a{};
  FFDP_TRY(make_geom(out_dims, mdims, T, a.g));
  a.M = M;
  a.u = u;
  a.gbuf = gJ;
  a.du = du;
  a.partials = reinterpret_cast<double*>(static_cast<char*>(ws) + w.partials);
  a.nIter = n_iter2(a.g.N, S2_GBUF);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = persistent_grid(a.nIter, sweep2_ctas_per_sm(S2_GBUF, 0, mt, 32));
  FFDP_CUDA(launch_sweep2(S2_GBUF, 0, mt, 32, a, grid, s), "grid_sample_bwd launch");
  if (dA || dt) {
    FinishArgs f{};
    f.partials = a.partials;
    f.nparts = grid;
    f.dA = dA;
    f.dt = dt;
    f.has_affine = 1;
    for (int c = 0; c < 3; ++c) {
      const double nf = c == 0 ? (double)out_dims.w : (c == 1 ? (double)out_dims.h : (double)out_dims.d);
      const double nmv = c == 0 ? (double)mdims.w : (c == 1 ? (double)mdims.h : (double)mdims.d);
      f.hM[c] = (nmv - 1.0) / 2.0;
      f.dx[c] = ((double)T->xmax[c] - (double)T->xmin[c]) / (nf - 1.0);
      f.xc[c] = (double)T->xmin[c] + f.dx[c] * (nf - 1.0) / 2.0;
    }
    FFDP_CUDA(launch_finish(f, s), "finish launch");
  }
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_mi_fwd_bwd(const void* F, ffdp_dtype ft, const float* J, ffdp_dims dims,
                                       const ffdp_mi_params* p, float* loss, float* dJ, void* ws,
                                       size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!F || !J || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null F, J or loss");
  FFDP_TRY(check_dtype(ft, "F"));
  FFDP_TRY(check_dims(dims, "image"));
  FFDP_TRY(check_mi(p));
  if (!aligned16(F) || !aligned16(J) || (dJ && !aligned16(dJ)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "F, J and dJ must be 16-byte aligned");
  const int bmax = bmax_of(p->bins);
  const Ws w = ws_layout(true, bmax, max_parts(), false, false, nvox(dims));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  char* wb = static_cast<char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Geom g;
  make_grid_only(dims, g);
  unsigned long long* hist = reinterpret_cast<unsigned long long*>(wb + w.hist);
  FFDP_CUDA(launch_zero_u64(hist, bmax * bmax, s), "zero launch");
  Sweep1Args a1{};
  a1.g = g;
  a1.F = F;
  a1.Jin = J;
  a1.ghist = hist;
  a1.bf = bin_map(p->f_lo, p->f_hi, p->bins);
  a1.bj = bin_map(p->m_lo, p->m_hi, p->bins);
  a1.B = p->bins;
  a1.nIter = n_iter1(g.N);
  FFDP_CUDA(launch_sweep1(S1_HIST_JBUF, ft, 0, bmax,
                          a1, persistent_grid(a1.nIter, sweep1_ctas_per_sm(S1_HIST_JBUF, ft, 0, bmax)), s),
            "MI histogram launch");
  FinalizeArgs fa{};
  fa.ghist = hist;
  fa.T = reinterpret_cast<float*>(wb + w.table);
  fa.scalars = reinterpret_cast<double*>(wb + w.scalars);
  fa.B = p->bins;
  fa.N = (double)g.N;
  fa.tscale = (double)(p->bins - 5) / ((double)p->m_hi - (double)p->m_lo) / (double)g.N;
  FFDP_CUDA(launch_finalize(bmax, fa, s), "MI finalize launch");
  if (dJ) {
    Sweep2Args a2{};
    a2.g = g;
    a2.F = F;
    a2.Jin = J;
    a2.dJ = dJ;
    a2.T = fa.T;
    a2.bf = a1.bf;
    a2.bj = a1.bj;
    a2.B = p->bins;
    a2.nIter = n_iter2(g.N, S2_MI_JBUF);
    FFDP_CUDA(launch_sweep2(S2_MI_JBUF, ft, 0, bmax, a2,
                            persistent_grid(a2.nIter, sweep2_ctas_per_sm(S2_MI_JBUF, ft, 0, bmax)), s),
              "MI gradient launch");
  }
  FinishArgs f{};
  f.scalars = fa.scalars;
  f.mi_rows = bmax;
  f.nparts = 0;
  f.partials = reinterpret_cast<double*>(wb + w.partials);
  f.loss = loss;
  f.nloss = 1;
  f.has_mi = 1;
  f.N = (double)g.N;
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_lncc_fwd_bwd(const void* F, ffdp_dtype ft, const float* J, ffdp_dims dims,
                                         const ffdp_lncc_params* p, float* loss, float* dJ, void* ws,
                                         size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!F || !J || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null F, J or loss");
  FFDP_TRY(check_dtype(ft, "F"));
  FFDP_TRY(check_dims(dims, "image"));
  FFDP_TRY(check_lncc(p));
  if (!aligned16(F) || !aligned16(J) || (dJ && !aligned16(dJ)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "F, J and dJ must be 16-byte aligned");
  const bool wide = lncc_wide(p->window);
  const Ws w = ws_layout(false, 32, max_parts(), false, false, nvox(dims), wide, lncc_split(p->window));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  char* wb = static_cast<char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (wide) {
    WideArgs a{};
    make_grid_only(dims, a.g);
    a.F = F;
    a.J = J;
    a.dJ = dJ;
    a.partials = reinterpret_cast<double*>(wb + w.partials);
    a.bufA = reinterpret_cast<float*>(wb + w.WA);
    a.bufB = reinterpret_cast<float*>(wb + w.WB);
    a.R = wide_radius(p->window, a.g);
    a.eps = p->eps;
    a.inv_n = (float)(1.0 / ((double)p->window * p->window * p->window));
    a.gscale = (float)(-1.0 / (double)a.g.N);
    const int grid = persistent_grid((unsigned)((a.g.N + 255) / 256), kWideCtasPerSm);
    FFDP_CUDA(launch_lncc_wide(LN_DJ, ft, 0, a, grid, s), "wide-window LNCC launch");
    FinishArgs f{};
    f.partials = a.partials;
    f.nparts = grid;
    f.loss = loss;
    f.nloss = 1;
    f.has_lncc = 1;
    f.N = (double)a.g.N;
    FFDP_CUDA(launch_finish(f, s), "finish launch");
    return FFDP_OK;
  }
  LnccArgs a{};
  make_grid_only(dims, a.g);
  a.F = F;
  a.J = J;
  a.dJ = dJ;
  a.gbuf = reinterpret_cast<float*>(wb + w.GS);
  a.partials = reinterpret_cast<double*>(wb + w.partials);
  a.R = (p->window - 1) / 2;
  a.eps = p->eps;
  a.inv_n = (float)(1.0 / ((double)p->window * p->window * p->window));
  a.gscale = (float)(-1.0 / (double)a.g.N);
  int grid = 1;
  lncc_tiling(dims, a.R, a, lncc_ctas_per_sm(LN_DJ, ft, 0, 0, a.R), grid);
  FFDP_CUDA(launch_lncc(LN_DJ, ft, 0, 0, a, grid, s), "LNCC launch");
  FinishArgs f{};
  f.partials = a.partials;
  f.nparts = grid;
  f.loss = loss;
  f.nloss = 1;
  f.has_lncc = 1;
  f.N = (double)a.g.N;
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

namespace {

// The objective pipeline of ffdp_objective (store_slope = false) and
// ffdp_objective_stored (store_slope = true: an MI-only objective keeps J and
// its slope for a streaming gradient pass).
ffdp_status objective(const void* F, ffdp_dtype ft, ffdp_dims fdims, const void* M, ffdp_dtype mt,
                      ffdp_dims mdims, const float* u, const ffdp_transform* T, const ffdp_objective_params* p,
                      float* loss, float* du, float* dA, float* dt, void* ws, size_t ws_bytes, void* stream,
                      bool store_slope) {
  g_err[0] = '\0';
  if (!F || !M || !T || !p || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null F, M, T, params or loss");
  FFDP_TRY(check_dtype(ft, "F"));
  FFDP_TRY(check_dtype(mt, "M"));
  FFDP_TRY(check_dims(fdims, "fixed"));
  FFDP_TRY(check_dims(mdims, "moving"));
  if (!std::isfinite(p->w_mi) || !std::isfinite(p->w_lncc))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "non-finite loss weights");
  const bool mi = p->w_mi != 0.0f, ln = p->w_lncc != 0.0f;
  if (!mi && !ln) return fail(FFDP_ERR_INVALID_ARGUMENT, "both loss weights are zero");
  if (mi) FFDP_TRY(check_mi(&p->mi));
  if (ln) FFDP_TRY(check_lncc(&p->lncc));
  if (ln && ft != mt) return fail(FFDP_ERR_UNSUPPORTED, "LNCC objective needs F and M of the same dtype");
  if (!aligned16(F) || (u && !aligned16(u)) || (du && !aligned16(du)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "F, u and du must be 16-byte aligned");
  const int bmax = mi ? bmax_of(p->mi.bins) : 32;
  const uint64_t N = nvox(fdims);
  const bool rc = ln && lncc_recompute(p->lncc.window);  // LNCC samples J on chip
  const bool store = (ln && !rc) || (mi && !ln && store_slope);
  const bool wide = ln && lncc_wide(p->lncc.window);
  const Ws w = ws_layout(mi, bmax, max_parts(), ln, store, N, wide, ln && lncc_split(p->lncc.window));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  char* wb = static_cast<char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Geom g;
  FFDP_TRY(make_geom(fdims, mdims, T, g));
  unsigned long long* hist = reinterpret_cast<unsigned long long*>(wb + w.hist);
  float* table = reinterpret_cast<float*>(wb + w.table);
  float* table2 = (mi && ln && bmax == 64) ? reinterpret_cast<float*>(wb + w.table2) : nullptr;
  double* scalars = reinterpret_cast<double*>(wb + w.scalars);
  double* partials = reinterpret_cast<double*>(wb + w.partials);
  float* Jbuf = store ? reinterpret_cast<float*>(wb + w.J) : nullptr;
  float* DGbuf = store ? reinterpret_cast<float*>(wb + w.DG) : nullptr;
  const BinMap bf = mi ? bin_map(p->mi.f_lo, p->mi.f_hi, p->mi.bins) : BinMap{0, 1, 1, 0};
  const BinMap bj = mi ? bin_map(p->mi.m_lo, p->mi.m_hi, p->mi.bins) : BinMap{0, 1, 1, 0};

  // sweep 1: histogram (MI) and/or the materialised J (LNCC); none for an
  // LNCC-only objective that samples J on chip
  if (mi) FFDP_CUDA(launch_zero_u64(hist, bmax * bmax, s), "zero launch");
  Sweep1Args a1{};
  a1.g = g;
  a1.F = F;
  a1.M = M;
  a1.u = u;
  a1.Jout = Jbuf;
  a1.Gout = DGbuf;
  a1.stall_tx = take_test_stall();
  a1.ghist = hist;
  a1.bf = bf;
  a1.bj = bj;
  a1.B = mi ? p->mi.bins : 32;
  a1.nIter = n_iter1(N);
  // with LNCC (or store_slope), J and its slope dJ/dq are stored for the
  // window kernel and the streaming gradient pass
  const int m1 = mi ? (store ? S1_HIST_WRITEJG : S1_HIST) : S1_WRITEJG;
  if (mi || !rc)
    FFDP_CUDA(launch_sweep1(m1, ft, mt, bmax, a1, persistent_grid(a1.nIter, sweep1_ctas_per_sm(m1, ft, mt, bmax)), s),
              "sweep 1 launch");
  if (mi) {
    FinalizeArgs fa{};
    fa.ghist = hist;
    fa.T = table;
    fa.T2 = table2;
    fa.scalars = scalars;
    fa.B = p->mi.bins;
    fa.N = (double)N;
    fa.tscale = (double)p->w_mi * (double)(p->mi.bins - 5) / ((double)p->mi.m_hi - (double)p->mi.m_lo) / (double)N;
    FFDP_CUDA(launch_finalize(bmax, fa, s), "MI finalize launch");
  }
  int nparts = 0;
  if (wide) {
    // wide window: separable box-sum passes, then g = dL/dJ (LNCC + MI term)
    // and the sampler backward from the stored slope
    WideArgs a{};
    a.g = g;
    a.F = F;
    a.J = Jbuf;
    a.dJdq = DGbuf;
    a.du = du;
    a.T = bmax == 64 ? table2 : table;
    a.partials = partials;
    a.bufA = reinterpret_cast<float*>(wb + w.WA);
    a.bufB = reinterpret_cast<float*>(wb + w.WB);
    a.bf = bf;
    a.bj = bj;
    a.R = wide_radius(p->lncc.window, g);
    a.eps = p->lncc.eps;
    a.inv_n = (float)(1.0 / ((double)p->lncc.window * p->lncc.window * p->lncc.window));
    a.gscale = (float)(-(double)p->w_lncc / (double)N);
    const int grid = persistent_grid((unsigned)((N + 255) / 256), kWideCtasPerSm);
    FFDP_CUDA(launch_lncc_wide(LN_DU, ft, mi ? bmax : 0, a, grid, s), "wide-window LNCC launch");
    nparts = grid;
  } else if (ln) {
    // LNCC window kernel: g = dL/dJ (LNCC term + MI term from on-chip J, F),
    // then the sampler backward from the stored slope (du, affine partials)
    LnccArgs a{};
    a.g = g;
    a.F = F;
    a.J = Jbuf;
    a.dJdq = DGbuf;
    a.M = M;
    a.u = u;
    a.du = du;
    a.gbuf = reinterpret_cast<float*>(wb + w.GS);
    a.T = bmax == 64 ? table2 : table;  // polynomial cells
    a.partials = partials;
    a.bf = bf;
    a.bj = bj;
    a.B = mi ? p->mi.bins : 0;
    a.R = (p->lncc.window - 1) / 2;
    a.eps = p->lncc.eps;
    a.inv_n = (float)(1.0 / ((double)p->lncc.window * p->lncc.window * p->lncc.window));
    a.gscale = (float)(-(double)p->w_lncc / (double)N);
    const int bm = mi ? bmax : 0;
    int grid = 1;
    lncc_tiling(fdims, a.R, a, lncc_ctas_per_sm(LN_DU, ft, 0, bm, a.R), grid);
    FFDP_CUDA(launch_lncc(LN_DU, ft, 0, bm, a, grid, s), "LNCC window launch");
    nparts = grid;
  } else {
    // MI gradient and sampler backward: gathers M again, or streams the stored J and slope
    const int m2 = store ? S2_MI_DJ : S2_MI;
    Sweep2Args a2{};
    a2.g = g;
    a2.F = F;
    a2.M = M;
    a2.u = u;
    a2.Jin = Jbuf;
    a2.dJdq = DGbuf;
    a2.du = du;
    a2.T = table;
    a2.partials = partials;
    a2.bf = bf;
    a2.bj = bj;
    a2.B = p->mi.bins;
    a2.nIter = n_iter2(N, m2);
    const int grid = persistent_grid(a2.nIter, sweep2_ctas_per_sm(m2, ft, mt, bmax));
    FFDP_CUDA(launch_sweep2(m2, ft, mt, bmax, a2, grid, s), "sweep 2 launch");
    nparts = grid;
  }
  FinishArgs f{};
  f.partials = partials;
  f.nparts = nparts;
  f.scalars = scalars;
  f.mi_rows = mi ? bmax : 0;
  f.dA = dA;
  f.dt = dt;
  f.loss = loss;
  f.nloss = 3;
  f.N = (double)N;
  f.w_mi = p->w_mi;
  f.w_lncc = p->w_lncc;
  f.has_mi = mi;
  f.has_lncc = ln;
  f.has_affine = 1;
  for (int c = 0; c < 3; ++c) {
    const double nf = c == 0 ? (double)fdims.w : (c == 1 ? (double)fdims.h : (double)fdims.d);
    const double nmv = c == 0 ? (double)mdims.w : (c == 1 ? (double)mdims.h : (double)mdims.d);
    f.hM[c] = (nmv - 1.0) / 2.0;
    f.dx[c] = ((double)T->xmax[c] - (double)T->xmin[c]) / (nf - 1.0);
    f.xc[c] = (double)T->xmin[c] + f.dx[c] * (nf - 1.0) / 2.0;
  }
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

}  // namespace

extern "C" ffdp_status ffdp_objective(const void* F, ffdp_dtype ft, ffdp_dims fdims, const void* M,
                                      ffdp_dtype mt, ffdp_dims mdims, const float* u,
                                      const ffdp_transform* T, const ffdp_objective_params* p, float* loss,
                                      float* du, float* dA, float* dt, void* ws, size_t ws_bytes,
                                      void* stream) {
  return objective(F, ft, fdims, M, mt, mdims, u, T, p, loss, du, dA, dt, ws, ws_bytes, stream, false);
}

extern "C" ffdp_status ffdp_objective_stored(const void* F, ffdp_dtype ft, ffdp_dims fdims, const void* M,
                                             ffdp_dtype mt, ffdp_dims mdims, const float* u,
                                             const ffdp_transform* T, const ffdp_objective_params* p,
                                             float* loss, float* du, float* dA, float* dt, void* ws,
                                             size_t ws_bytes, void* stream) {
  return objective(F, ft, fdims, M, mt, mdims, u, T, p, loss, du, dA, dt, ws, ws_bytes, stream, true);
}

// ------------------------------------------- C-channel sampler (composition)
namespace {

ffdp_status check_channels(const float* V, int C, ffdp_dims vdims, ffdp_dims out_dims, int compose) {
  if (!V) return fail(FFDP_ERR_INVALID_ARGUMENT, "null V");
  if (C < 1 || C > 4) return fail(FFDP_ERR_INVALID_ARGUMENT, "channels must be in [1, 4] (got %d)", C);
  if (compose && C != 3) return fail(FFDP_ERR_INVALID_ARGUMENT, "compose needs a 3-channel displacement field V");
  FFDP_TRY(check_dims(vdims, "V"));
  FFDP_TRY(check_dims(out_dims, "output"));
  if (!aligned16(V)) return fail(FFDP_ERR_INVALID_ARGUMENT, "V must be 16-byte aligned");
  return FFDP_OK;
}

void fill_finish_affine(FinishArgs& f, ffdp_dims fdims, ffdp_dims mdims, const ffdp_transform* T) {
  for (int c = 0; c < 3; ++c) {
    const double nf = c == 0 ? (double)fdims.w : (c == 1 ? (double)fdims.h : (double)fdims.d);
    const double nmv = c == 0 ? (double)mdims.w : (c == 1 ? (double)mdims.h : (double)mdims.d);
    f.hM[c] = (nmv - 1.0) / 2.0;
    f.dx[c] = ((double)T->xmax[c] - (double)T->xmin[c]) / (nf - 1.0);
    f.xc[c] = (double)T->xmin[c] + f.dx[c] * (nf - 1.0) / 2.0;
  }
}

int chan_grid(uint64_t N, int C, int compose, int bwd) {
  const uint64_t ctas = (N + kChanThreads - 1) / kChanThreads;
  const uint64_t slots = (uint64_t)(sm_count() > 0 ? sm_count() : 1) * chan_ctas_per_sm(C, compose, bwd);
  return (int)(ctas < slots ? (ctas < 1 ? 1 : ctas) : slots);
}

}  // namespace

extern "C" ffdp_status ffdp_sample_channels_fwd(const float* V, int C, ffdp_dims vdims, ffdp_dims out_dims,
                                                const float* u, const ffdp_transform* T, int compose, float* out,
                                                void* stream) {
  g_err[0] = '\0';
  if (!T || !out) return fail(FFDP_ERR_INVALID_ARGUMENT, "null T or out");
  FFDP_TRY(check_channels(V, C, vdims, out_dims, compose));
  if (!aligned16(out) || (u && !aligned16(u))) return fail(FFDP_ERR_INVALID_ARGUMENT, "out and u must be 16-byte aligned");
  ChanArgs a{};
  FFDP_TRY(make_geom(out_dims, vdims, T, a.g));
  a.V = V;
  a.u = u;
  a.out = out;
  for (int k = 0; k < 9; ++k) a.S[k] = T->S[k];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FFDP_CUDA(launch_chan_fwd(C, compose, a, chan_grid(a.g.N, C, compose, 0), s), "channel sampler launch");
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_sample_channels_bwd(const float* V, int C, ffdp_dims vdims, ffdp_dims out_dims,
                                                const float* u, const ffdp_transform* T, int compose,
                                                const float* gout, float* du, float* dA, float* dt, float* dV,
                                                void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!T || !gout) return fail(FFDP_ERR_INVALID_ARGUMENT, "null T or gout");
  FFDP_TRY(check_channels(V, C, vdims, out_dims, compose));
  if ((u && !aligned16(u)) || !aligned16(gout) || (du && !aligned16(du)) || (dV && !aligned16(dV)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "u, gout, du and dV must be 16-byte aligned");
  const Ws w = ws_layout(false, 32, max_parts(), false, false, nvox(out_dims));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  ChanArgs a{};
  FFDP_TRY(make_geom(out_dims, vdims, T, a.g));
  a.V = V;
  a.u = u;
  a.gout = gout;
  a.du = du;
  a.dV = dV;
  a.partials = reinterpret_cast<double*>(static_cast<char*>(ws) + w.partials);
  a.nV = (long long)nvox(vdims) * C;
  for (int k = 0; k < 9; ++k) a.S[k] = T->S[k];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dV) FFDP_CUDA(launch_zero_f32(dV, a.nV, s), "dV zero launch");
  const int grid = chan_grid(a.g.N, C, compose, 1);
  FFDP_CUDA(launch_chan_bwd(C, compose, a, grid, s), "channel sampler backward launch");
  if (dA || dt) {
    FinishArgs f{};
    f.partials = a.partials;
    f.nparts = grid;
    f.dA = dA;
    f.dt = dt;
    f.has_affine = 1;
    fill_finish_affine(f, out_dims, vdims, T);
    FFDP_CUDA(launch_finish(f, s), "finish launch");
  }
  return FFDP_OK;
}

// ------------------------------------------------------------------- MSE
extern "C" ffdp_status ffdp_mse_fwd_bwd(const void* F, ffdp_dtype ft, const float* J, ffdp_dims dims, float* loss,
                                        float* dJ, void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!F || !J || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null F, J or loss");
  FFDP_TRY(check_dtype(ft, "F"));
  FFDP_TRY(check_dims(dims, "image"));
  if (!aligned16(F) || !aligned16(J) || (dJ && !aligned16(dJ)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "F, J and dJ must be 16-byte aligned");
  const Ws w = ws_layout(false, 32, max_parts(), false, false, nvox(dims));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MseArgs a{};
  a.F = F;
  a.J = J;
  a.dJ = dJ;
  a.partials = reinterpret_cast<double*>(static_cast<char*>(ws) + w.partials);
  a.N = (unsigned)nvox(dims);
  a.c = (float)(2.0 / (double)a.N);
  const int grid = chan_grid((a.N + 3) / 4, 0, 0, 0);
  FFDP_CUDA(launch_mse(ft, a, grid, s), "MSE launch");
  FinishArgs f{};
  f.partials = a.partials;
  f.nparts = grid;
  f.loss = loss;
  f.nloss = 1;
  f.has_mse = 1;
  f.w_mse = 1.0;
  f.N = (double)a.N;
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

extern "C" ffdp_status ffdp_objective_mse(const void* F, ffdp_dtype ft, ffdp_dims fdims, const void* M,
                                          ffdp_dtype mt, ffdp_dims mdims, const float* u, const ffdp_transform* T,
                                          float w_mse, float* loss, float* du, float* dA, float* dt, void* ws,
                                          size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!F || !M || !T || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null F, M, T or loss");
  FFDP_TRY(check_dtype(ft, "F"));
  FFDP_TRY(check_dtype(mt, "M"));
  FFDP_TRY(check_dims(fdims, "fixed"));
  FFDP_TRY(check_dims(mdims, "moving"));
  if (!std::isfinite(w_mse) || w_mse == 0.0f) return fail(FFDP_ERR_INVALID_ARGUMENT, "w_mse must be finite and non-zero");
  if (!aligned16(F) || (u && !aligned16(u)) || (du && !aligned16(du)))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "F, u and du must be 16-byte aligned");
  const uint64_t N = nvox(fdims);
  const Ws w = ws_layout(false, 32, max_parts(), false, false, N);
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Sweep2Args a2{};
  FFDP_TRY(make_geom(fdims, mdims, T, a2.g));
  a2.F = F;
  a2.M = M;
  a2.u = u;
  a2.du = du;
  a2.partials = reinterpret_cast<double*>(static_cast<char*>(ws) + w.partials);
  a2.mse_c = (float)(2.0 * (double)w_mse / (double)N);
  a2.nIter = n_iter2(N, S2_MSE);
  const int grid = persistent_grid(a2.nIter, sweep2_ctas_per_sm(S2_MSE, ft, mt, 32));
  FFDP_CUDA(launch_sweep2(S2_MSE, ft, mt, 32, a2, grid, s), "MSE sweep launch");
  FinishArgs f{};
  f.partials = a2.partials;
  f.nparts = grid;
  f.dA = dA;
  f.dt = dt;
  f.loss = loss;
  f.nloss = 2;
  f.N = (double)N;
  f.w_mse = w_mse;
  f.has_mse = 1;
  f.has_affine = 1;
  fill_finish_affine(f, fdims, mdims, T);
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

// -------------------------------------- Sobolev regulariser, Adam step of u
namespace {

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

ffdp_status reg_launch(int step, RegArgs& a, ffdp_dims dims, float* loss, void* ws, size_t ws_bytes, void* stream) {
  const Ws w = ws_layout(false, 32, max_parts(), false, false, nvox(dims));
  FFDP_TRY(check_ws(ws, ws_bytes, w.total));
  make_grid_only(dims, a.g3);
  a.partials = reinterpret_cast<double*>(static_cast<char*>(ws) + w.partials);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t N = nvox(dims);
  const uint64_t groups = (N + 31) / 32;
  const uint64_t ctas = (groups + kRegThreads / 32 - 1) / (kRegThreads / 32);
  const uint64_t slots = (uint64_t)(sm_count() > 0 ? sm_count() : 1) * reg_ctas_per_sm(step);
  const int grid = (int)(ctas < slots ? (ctas < 1 ? 1 : ctas) : slots);
  FFDP_CUDA(launch_reg(step, a, grid, s), "regulariser launch");
  FinishArgs f{};
  f.partials = a.partials;
  f.nparts = grid;
  f.loss = loss;
  f.nloss = 1;
  f.has_mse = 1;  // the per-CTA slot holds lambda * sum of squares: loss = that / N
  f.w_mse = 1.0;
  f.N = (double)N;
  FFDP_CUDA(launch_finish(f, s), "finish launch");
  return FFDP_OK;
}

}  // namespace

extern "C" ffdp_status ffdp_sobolev_fwd_bwd(const float* u, ffdp_dims dims, float lambda, float* loss, float* dR,
                                            void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!u || !loss) return fail(FFDP_ERR_INVALID_ARGUMENT, "null u or loss");
  FFDP_TRY(check_dims(dims, "u"));
  if (!std::isfinite(lambda) || lambda < 0.0f) return fail(FFDP_ERR_INVALID_ARGUMENT, "lambda must be finite and >= 0");
  if (!aligned16(u) || (dR && !aligned16(dR))) return fail(FFDP_ERR_INVALID_ARGUMENT, "u and dR must be 16-byte aligned");
  const size_t bytes = (size_t)nvox(dims) * 12;
  if (dR && overlaps(u, bytes, dR, bytes)) return fail(FFDP_ERR_INVALID_ARGUMENT, "dR must not overlap u");
  RegArgs a{};
  a.u = u;
  a.dR = dR;
  a.lambda = lambda;
  a.coef = (float)(2.0 * (double)lambda / (double)nvox(dims));
  return reg_launch(0, a, dims, loss, ws, ws_bytes, stream);
}

extern "C" ffdp_status ffdp_sobolev_adam_step(const float* u, float* u_out, const float* g, float* m1, float* m2,
                                              ffdp_dims dims, const ffdp_sobolev_adam_params* p, float* loss,
                                              void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = '\0';
  if (!u || !u_out || !g || !m1 || !m2 || !p || !loss)
    return fail(FFDP_ERR_INVALID_ARGUMENT, "null u, u_out, g, m1, m2, params or loss");
  FFDP_TRY(check_dims(dims, "u"));
  if (!aligned16(u) || !aligned16(u_out) || !aligned16(g) || !aligned16(m1) || !aligned16(m2))
    return fail(FFDP_ERR_INVALID_ARGUMENT, "u, u_out, g, m1 and m2 must be 16-byte aligned");
  const size_t bytes = (size_t)nvox(dims) * 12;
  if (overlaps(u, bytes, u_out, bytes)) return fail(FFDP_ERR_INVALID_ARGUMENT, "u_out must not overlap u");
  if (overlaps(m1, bytes, m2, bytes)) return fail(FFDP_ERR_INVALID_ARGUMENT, "m1 and m2 must not overlap");
  if (!std::isfinite(p->lambda) || p->lambda < 0.0f || !std::isfinite(p->lr) || !(p->beta1 >= 0.0f && p->beta1 < 1.0f) ||
      !(p->beta2 >= 0.0f && p->beta2 < 1.0f) || !std::isfinite(p->eps) || p->eps < 0.0f || p->step < 1)
    return fail(FFDP_ERR_INVALID_ARGUMENT,
                "need finite lambda >= 0, finite lr, beta1 and beta2 in [0, 1), eps >= 0 and step >= 1");
  RegArgs a{};
  a.u = u;
  a.g = g;
  a.u_out = u_out;
  a.m1 = m1;
  a.m2 = m2;
  a.lambda = p->lambda;
  a.coef = (float)(2.0 * (double)p->lambda / (double)nvox(dims));
  a.lr = p->lr;
  a.b1 = p->beta1;
  a.b2 = p->beta2;
  a.eps = p->eps;
  a.ic1 = (float)(1.0 / (1.0 - std::pow((double)p->beta1, (double)p->step)));
  a.ic2 = (float)(1.0 / (1.0 - std::pow((double)p->beta2, (double)p->step)));
  return reg_launch(1, a, dims, loss, ws, ws_bytes, stream);
}

// ------------------------------------------------ workspace-free MI objective
// Some callers cannot hand the library a workspace: a plug-in running inside a
// host application that owns every device allocation, a real-time loop whose
// rules forbid allocating after start-up, or a plain C host that only holds
// its input and output buffers and has no device allocator of its own.  For
// them the MI-only objective can run on scratch memory reserved inside the
// library image: this file-scope array is created on every GPU that loads the
// library and is held until the process exits.  Host code must not use the
// array's name as a device address (in host code it is only a stand-in): the
// device address is looked up with cudaGetSymbolAddress, with the caller's
// device current, and passed to the kernels.  The lookup is repeated on every
// call (after the first call on a device, which loads the module, it is a
// table lookup in the runtime), so an address never outlives the context it
// belongs to: after a cudaDeviceReset the next call finds the array again in
// the new context.
static constexpr size_t kStaticScratchBytes = 512u * 1024u;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
ffdp_status static_scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  *out = p;
  return FFDP_OK;
}
}  // namespace

extern "C" size_t ffdp_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" ffdp_status ffdp_objective_mi_static(const void* F, ffdp_dtype ft, ffdp_dims fdims, const void* M,
                                                ffdp_dtype mt, ffdp_dims mdims, const float* u,
                                                const ffdp_transform* T, const ffdp_objective_params* p,
                                                float* loss, float* du, float* dA, float* dt, void* stream) {
  g_err[0] = '\0';
  if (!p) return fail(FFDP_ERR_INVALID_ARGUMENT, "null params");
  if (p->w_lncc != 0.0f)
    return fail(FFDP_ERR_UNSUPPORTED,
                "the workspace-free objective evaluates MI only (w_lncc must be 0): LNCC keeps a "
                "per-voxel image that does not fit the %zu-byte static scratch",
                kStaticScratchBytes);
  const size_t need = ffdp_workspace_bytes(FFDP_OP_OBJECTIVE, fdims, p);
  if (need == 0) {
    if (g_err[0] == '\0') fail(FFDP_ERR_INVALID_ARGUMENT, "invalid objective parameters or dimensions");
    return FFDP_ERR_INVALID_ARGUMENT;
  }
  if (need > kStaticScratchBytes)
    return fail(FFDP_ERR_UNSUPPORTED, "this call needs %zu bytes of scratch; the static scratch holds %zu",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  FFDP_TRY(static_scratch_address(&scratch));
  return ffdp_objective(F, ft, fdims, M, mt, mdims, u, T, p, loss, du, dA, dt, scratch, kStaticScratchBytes,
                        stream);
}
