// C-ABI layer of the RankMixer library: argument checks, the layout of the
// saved and scratch buffers, and the launch sequences of the forward and
// backward passes (all on the caller's stream; nothing here allocates device
// memory or synchronises, except rmx_check and rmx_profile_read).
//
// Forward (page "Subgraph-fusion-based Mega-kernel Generation", section
// "Exact computation"):
//   1. norm0 -> token mix -> + x -> norm1          -> out1        (row pass)
//   2. Z = out1[:,t] @ w1[t] + b1[t]                -> Z           (GEMM, bias)
//   3. hidden = LN_x(U) * silu(LN_gate(G))          -> hidden      (row pass)
//   4. s2 = hidden[:,t] @ wout[t] + bout[t] + out1  -> s2          (GEMM, bias+residual)
//   5. y = norm2(s2)                                               (row pass)
// Backward (chain rule through the same steps, in reverse):
//   1. ds2 = norm2-backward(dy), partials of dgamma2/dbeta2/dbout
//   2. dh = ds2[:,t] @ wout[t]^T                                   (GEMM, NT)
//   3. dwout[t] = hidden[:,t]^T @ ds2[:,t]                         (GEMM, TN)
//   4. dZ = gate/inner-LN backward(dh), partials of their params and db1
//   5. dout1 = dZ[:,t] @ w1[t]^T + ds2                             (GEMM, NT, residual)
//   6. dw1[t] = out1[:,t]^T @ dZ[:,t]                              (GEMM, TN)
//   7. dx = norm1/mix/norm0 backward(dout1), partials of their params
//   8. fixed-order column sums of every partial
// The backward is launched on the caller's stream in the order 1 2 4 5 7 3 6
// 8: the weight gradients, which nothing else consumes, come last.

#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/rmx.h"
#include "common.cuh"
#include "kernels.h"

namespace rmx {

__device__ unsigned int g_rmx_error_word;

unsigned int* device_error_word() {
  // Per-device address, cached; several host threads may look it up at once
  // (they all store the same value).
  static std::atomic<unsigned int*> addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned int* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rmx_error_word) != cudaSuccess) return nullptr;
    a = static_cast<unsigned int*>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline int esize(int dtype) { return dtype == RMX_F32 || dtype == RMX_F32_TF32 ? 4 : 2; }
// Storage type of a config's tensors: the TF32 contract stores fp32.
inline int storage(int dtype) { return dtype == RMX_F32_TF32 ? RMX_F32 : dtype; }

// ------------------------------------------------------------------ layouts
constexpr int kNumParams = 14;

// Offsets of the 14 parameter-shaped tensors (rmx_params order) in a buffer.
struct ParamSet {
  size_t off[kNumParams];
};

struct Layout {
  // Row pitches the kernels see (multiples of 8) and the block's own sizes.
  // When they differ, the block runs on zero-padded copies (`padded`).
  int D, H, Dl, Hl;
  bool padded;
  // saved (filled by the forward)
  size_t out1, Z, hidden, s2, stats, zstats, s1, saved_total;
  // padded copies of x, y and the parameters (in `saved`), of dy, dx and
  // the gradients (in `ws`)
  size_t xp, yp, dyp, dxp;
  ParamSet pp, gp;
  // TF32 contract: K-major (transposed) copies of the operands the
  // contractions read MN-major: w1, wout (saved), and hidden, ds2, out1, dZ
  // with the batch as the contraction axis padded to Bp (scratch).
  size_t w1T, woutT, hT, ds2T, out1T, dZT;
  int Bp;
  // backward scratch
  size_t ds2, dh, dZ, dout1, ds1, da0, pg2, pb2, pbo, pwx, pbx, pwg, pbg, pb1, pg0, pb0, pg1, pbe1, ws_total;
  RowArgs ra;
};

inline int pad8(int v) { return (v + 7) / 8 * 8; }

// Logical and padded shape of each parameter, in rmx_params order: rows x
// cols per outer index (w1 and b1 have their columns split into the U and G
// halves).
PadMap param_map(int k, int T, int D, int H, int Dp, int Hp) {
  switch (k) {
    case 0: return PadMap{T, D, Dp, 2 * H, 2 * Hp, 2};   // w1 [T, D, 2H]
    case 1: return PadMap{1, T, T, 2 * H, 2 * Hp, 2};    // b1 [T, 2H]
    case 2: return PadMap{T, H, Hp, D, Dp, 1};           // wout [T, H, D]
    case 3: return PadMap{1, T, T, D, Dp, 1};            // bout [T, D]
    default:
      if (k < 10) return PadMap{1, 1, 1, D, Dp, 1};      // outer LayerNorms [D]
      return PadMap{1, 1, 1, H, Hp, 1};                  // inner LayerNorms [H]
  }
}

size_t lay_params(size_t o, int T, int Dp, int Hp, size_t e, ParamSet& ps, size_t (*up)(size_t)) {
  for (int k = 0; k < kNumParams; ++k) {
    const PadMap m = param_map(k, T, Dp, Hp, Dp, Hp);
    ps.off[k] = o;
    o = up(o + (size_t)m.outer * m.rows_p * m.cols_p * e);
  }
  return o;
}

bool config_ok(const rmx_config* c) {
  if (!c) return false;
  if (c->B < 0 || c->T < 1 || c->D < 1 || c->H < 1) return false;
  if (c->D % c->T) return false;
  if (c->dtype != RMX_F32 && c->dtype != RMX_BF16 && c->dtype != RMX_F16 && c->dtype != RMX_F32_TF32) return false;
  const long long rows = (long long)c->B * c->T;
  if (rows > (1ll << 30) || (long long)c->D > (1 << 20) || (long long)c->H > (1 << 20)) return false;
  return true;
}

constexpr int kColsumJobs = 12;

// Rows per CTA (at most max_rows) for a grid of T x ceil(B / nb) CTAs of
// which `slots` are resident at once: the one with the shortest estimated
// run, (waves, rounded up) x (nb + overhead), where `overhead` is a CTA's
// fixed cost in rows (its prologue, ring fill and partial-sum writes); among
// equals the largest nb (fewer CTAs and partial rows).  A grid that is a
// whole number of waves wastes no tail.
int rows_per_cta(int B, int T, int slots, int max_rows, int overhead) {
  if (B <= 0) return 1;
  if (slots < 1) slots = 1;
  int best = 1;
  long long best_cost = -1;
  for (int nb = max_rows < B ? max_rows : B; nb >= 1; --nb) {
    const long long blocks = (B + nb - 1) / nb;
    const long long waves = ((long long)T * blocks + slots - 1) / slots;
    const long long cost = waves * (nb + overhead);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = nb;
    }
  }
  return best;
}
void colsum_jobs(const Layout& L, const rmx_config& c, const rmx_grads* g, void* ws, ColsumJob* jobs);

Layout layout_of(const rmx_config& c) {
  Layout L;
  L.Dl = c.D;
  L.Hl = c.H;
  L.D = pad8(c.D);
  L.H = pad8(c.H);
  L.padded = L.D != L.Dl || L.H != L.Hl;
  const size_t e = esize(c.dtype);
  const size_t N = (size_t)c.B * c.T, D = L.D, H = L.H;
  size_t o = 0;
  L.out1 = o; o = up(o + N * D * e);
  L.Z = o; o = up(o + N * 2 * H * e);
  L.hidden = o; o = up(o + N * H * e);
  L.s2 = o; o = up(o + N * D * e);
  L.stats = o; o = up(o + 10 * N * sizeof(float));
  L.zstats = o; o = up(o + N * (size_t)zstats_tiles(L.H) * 4 * sizeof(float));  // forward scratch
  L.s1 = o; o = up(o + N * D * e);  // norm1's input token_mix(norm0(x)) + x, read by its backward
  L.xp = L.yp = 0;
  if (L.padded) {
    L.xp = o; o = up(o + N * D * e);
    L.yp = o; o = up(o + N * D * e);
    o = lay_params(o, c.T, L.D, L.H, e, L.pp, up);
  }
  const bool tf32 = c.dtype == RMX_F32_TF32;
  const size_t T = c.T;
  L.w1T = L.woutT = L.hT = L.ds2T = L.out1T = L.dZT = 0;
  L.Bp = (c.B + 3) / 4 * 4;
  if (tf32) {
    L.w1T = o; o = up(o + T * 2 * H * D * e);
    L.woutT = o; o = up(o + T * D * H * e);
  }
  L.saved_total = o;

  L.ra.B = c.B;
  L.ra.T = c.T;
  L.ra.D = L.D;
  L.ra.H = L.H;
  L.ra.Dl = L.Dl;
  L.ra.Hl = L.Hl;
  L.ra.dtype = storage(c.dtype);
  // Rows per CTA of the per-token row passes (grid T x ceil(B / nb)).
  const int sms = c.B > 0 ? sm_count() : 1;
  // A gate CTA also loads the four weight vectors and writes six column
  // partials of H floats (about eight rows' worth of traffic); a LayerNorm
  // ring CTA writes two or three partial rows of D floats, which the column
  // sums read back (about four rows' worth).
  const int nb = rows_per_cta(c.B, c.T, sms * (c.B > 0 ? gate_bwd_ctas_per_sm(L.ra) : 1), kGateBwdMaxRows, 8);
  L.ra.nb = nb;
  L.ra.nbblk = c.B > 0 ? (c.B + nb - 1) / nb : 0;
  const int nbl = rows_per_cta(c.B, c.T, sms * (c.B > 0 ? ln_bwd_ctas_per_sm(L.ra) : 1), kLnBwdMaxRows, 4);
  L.ra.nb_ln = nbl;
  L.ra.nbblk_ln = c.B > 0 ? (c.B + nbl - 1) / nbl : 0;
  const size_t P = (size_t)L.ra.nbblk * c.T;     // gate-backward partial rows
  const size_t PL = (size_t)L.ra.nbblk_ln * c.T; // LayerNorm-backward partial rows
  const size_t P0 = ln0_bwd_gather_supported(L.ra) ? (size_t)ln0_bwd_partial_rows(L.ra) : PL;  // norm0's

  o = 0;
  L.ds2 = o; o = up(o + N * D * e);
  // dh, then (once the gate backward has consumed it) dout1, then ds1 in
  // place of dout1 (norm1's backward reads each row before writing it).
  L.dh = o; o = up(o + N * (H > D ? H : D) * e);
  L.dout1 = L.dh;
  L.ds1 = L.dh;
  L.dZ = o; o = up(o + N * 2 * H * e);
  L.da0 = o;  // token_mix(ds1): only when norm0's backward cannot gather it
  if (!ln0_bwd_gather_supported(L.ra)) o = up(o + N * D * e);
  L.pg2 = o; o = up(o + PL * D * sizeof(float));
  L.pb2 = o; o = up(o + PL * D * sizeof(float));
  L.pbo = o; o = up(o + PL * D * sizeof(float));
  L.pwx = o; o = up(o + P * H * sizeof(float));
  L.pbx = o; o = up(o + P * H * sizeof(float));
  L.pwg = o; o = up(o + P * H * sizeof(float));
  L.pbg = o; o = up(o + P * H * sizeof(float));
  L.pb1 = o; o = up(o + P * 2 * H * sizeof(float));
  L.pg0 = o; o = up(o + P0 * D * sizeof(float));
  L.pb0 = o; o = up(o + P0 * D * sizeof(float));
  L.pg1 = o; o = up(o + PL * D * sizeof(float));
  L.pbe1 = o; o = up(o + PL * D * sizeof(float));
  L.dyp = L.dxp = 0;
  if (L.padded) {
    L.dyp = o; o = up(o + N * D * e);
    L.dxp = o; o = up(o + N * D * e);
    o = lay_params(o, c.T, L.D, L.H, e, L.gp, up);
  }
  if (tf32) {
    const size_t Bp = L.Bp;
    L.hT = o; o = up(o + T * H * Bp * e);
    L.ds2T = o; o = up(o + T * D * Bp * e);
    L.out1T = o; o = up(o + T * D * Bp * e);
    L.dZT = o; o = up(o + T * 2 * H * Bp * e);
  }
  L.ws_total = o;
  return L;
}

// The backward's column-sum jobs: every partial buffer of `ws` and the
// gradient it reduces into (both null when only the sizes are wanted).
void colsum_jobs(const Layout& L, const rmx_config& c, const rmx_grads* g, void* ws, ColsumJob* jobs) {
  auto F = [&](size_t off) { return ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + off) : nullptr; };
  const int P = L.ra.nbblk * c.T, Pb = L.ra.nbblk;
  const int PL = L.ra.nbblk_ln * c.T, PLb = L.ra.nbblk_ln;
  const int P0 = ln0_bwd_gather_supported(L.ra) ? ln0_bwd_partial_rows(L.ra) : PL;
  const int D = L.D, H = L.H;
  const ColsumJob j[kColsumJobs] = {
      {F(L.pg2), g ? g->gamma2 : nullptr, PL, D},  {F(L.pb2), g ? g->beta2 : nullptr, PL, D},
      {F(L.pbo), g ? g->bout : nullptr, PLb, c.T * D}, {F(L.pwx), g ? g->lnx_w : nullptr, P, H},
      {F(L.pbx), g ? g->lnx_b : nullptr, P, H},    {F(L.pwg), g ? g->lng_w : nullptr, P, H},
      {F(L.pbg), g ? g->lng_b : nullptr, P, H},    {F(L.pb1), g ? g->b1 : nullptr, Pb, c.T * 2 * H},
      {F(L.pg1), g ? g->gamma1 : nullptr, PL, D},  {F(L.pbe1), g ? g->beta1 : nullptr, PL, D},
      {F(L.pg0), g ? g->gamma0 : nullptr, P0, D},  {F(L.pb0), g ? g->beta0 : nullptr, P0, D},
  };
  for (int k = 0; k < kColsumJobs; ++k) jobs[k] = j[k];
}

// What the kernels can do (beyond what makes a valid block).  Rows of any
// length run on copies padded to a multiple of 8 elements; the limits are on
// the padded lengths.
rmx_status kernels_support(const rmx_config& c) {
  const int V = 16 / esize(c.dtype);
  const Layout L = layout_of(c);
  if (L.D / V > kRowThreadsMax) return RMX_ERR_UNSUPPORTED;     // LN backward: a thread per 16-byte vector
  if ((L.D / V + 31) / 32 > 10) return RMX_ERR_UNSUPPORTED;  // LN forward: 10 vectors per lane
  if (!gate_bwd_fused_supported(L.ra)) return RMX_ERR_UNSUPPORTED;  // gate backward: 8 columns per thread
  return RMX_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rmx_status check_params(const rmx_params* p) {
  if (!p) return RMX_ERR_INVALID_ARG;
  const void* v[] = {p->w1, p->b1, p->wout, p->bout, p->gamma0, p->beta0, p->gamma1,
                     p->beta1, p->gamma2, p->beta2, p->lnx_w, p->lnx_b, p->lng_w, p->lng_b};
  for (const void* q : v) {
    if (!q) return RMX_ERR_INVALID_ARG;
    if (!aligned16(q)) return RMX_ERR_ALIGNMENT;
  }
  return RMX_OK;
}

rmx_status check_grads(const rmx_grads* g) {
  if (!g) return RMX_ERR_INVALID_ARG;
  void* v[] = {g->w1, g->b1, g->wout, g->bout, g->gamma0, g->beta0, g->gamma1,
               g->beta1, g->gamma2, g->beta2, g->lnx_w, g->lnx_b, g->lng_w, g->lng_b};
  for (void* q : v) {
    if (!q) return RMX_ERR_INVALID_ARG;
    if (!aligned16(q)) return RMX_ERR_ALIGNMENT;
  }
  return RMX_OK;
}

rmx_status check_ptr(const void* p) {
  if (!p) return RMX_ERR_INVALID_ARG;
  if (!aligned16(p)) return RMX_ERR_ALIGNMENT;
  return RMX_OK;
}

// ------------------------------------------------------------------ instrumentation
std::atomic<long long> g_launches{0};
std::atomic<bool> g_prof{false};
std::mutex g_mu;
std::string g_prof_only;  // when not empty, only launches of this name are timed (under g_mu)
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t pool_event() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

bool selected(const char* name) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_prof_only.empty() || g_prof_only == name;
}

// Brackets one kernel launch: counts it and, when profiling is on (for its
// name), records events around it on its stream.
class Launch {
 public:
  Launch(const char* name, cudaStream_t st) : name_(name), st_(st) {
    if (g_prof.load() && selected(name)) {
      a_ = pool_event();
      if (a_) cudaEventRecord(a_, st_);
    }
  }
  rmx_status done(cudaError_t e) {
    g_launches.fetch_add(1);
    if (a_) {
      cudaEvent_t b = pool_event();
      if (b) {
        cudaEventRecord(b, st_);
        std::lock_guard<std::mutex> lk(g_mu);
        g_recs.push_back({name_, a_, b});
      }
    }
    return e == cudaSuccess ? RMX_OK : RMX_ERR_CUDA;
  }

 private:
  const char* name_;
  cudaStream_t st_;
  cudaEvent_t a_ = nullptr;
};

#define RMX_TRY(expr)                  \
  do {                                 \
    rmx_status s_ = (expr);            \
    if (s_ != RMX_OK) return s_;       \
  } while (0)

// Profile name of a GEMM that runs on the CUDA cores (the strict fp32
// contract, or a 16-bit shape the tensor-core engine does not take).
const char* ffma_label(const char* name) {
  static const char* const kNames[][2] = {
      {"gemm1_fwd", "gemm1_fwd.ffma"},     {"gemm2_fwd", "gemm2_fwd.ffma"},
      {"gemm1_dgrad", "gemm1_dgrad.ffma"}, {"gemm2_dgrad", "gemm2_dgrad.ffma"},
      {"gemm1_wgrad", "gemm1_wgrad.ffma"}, {"gemm2_wgrad", "gemm2_wgrad.ffma"},
      {"test_gemm", "test_gemm.ffma"},
  };
  for (const auto& n : kNames)
    if (std::strcmp(n[0], name) == 0) return n[1];
  return name;
}

// Whether a contraction runs on the tensor cores: 16-bit storage, or fp32
// under the TF32 contract; otherwise (the strict fp32 contract) on the CUDA
// cores.
bool tc_engine(const GemmDesc& d) { return (d.dtype != RMX_F32 || d.tf32) && gemm_tc_supported(d); }

rmx_status run_gemm(const char* name, const GemmDesc& d, cudaStream_t st) {
  const bool tc = tc_engine(d);
  Launch l(tc ? name : ffma_label(name), st);
  const cudaError_t e = tc ? gemm_tc_launch(d, device_error_word(), st) : gemm_simt_launch(d, st);
  return l.done(e);
}

// Copy stream of rmx_step_host, one per device, created on first use; the
// events are shared, so a call's enqueue sequence holds g_copy_mu.
// x is uploaded in this many chunks of samples, so that the per-sample
// norm0/norm1 pass starts on the first chunks while the rest is in flight.
constexpr int kXChunks = 4;
// Sample ranges of the forward in rmx_step_host: two measured faster end to
// end than one (the upload of x no longer precedes all of the forward) and
// than four (each range reads the weights again).
constexpr int kFwdChunks = 2;

struct CopyStream {
  cudaStream_t s = nullptr;
  cudaEvent_t start = nullptr, dy_in = nullptr, fwd_done = nullptr, dx_ready = nullptr, done = nullptr;
  cudaEvent_t x_in[kXChunks] = {};
};
std::mutex g_copy_mu;

CopyStream* copy_stream() {
  static CopyStream cs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  CopyStream& c = cs[dev];
  if (!c.s) {
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    cudaEvent_t* ev[5] = {&c.start, &c.dy_in, &c.fwd_done, &c.dx_ready, &c.done};
    for (cudaEvent_t* e : ev)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    for (cudaEvent_t& e : c.x_in)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    c.s = s;
  }
  return &c;
}

inline char* at(void* base, size_t off) { return static_cast<char*>(base) + off; }
inline const char* at(const void* base, size_t off) { return static_cast<const char*>(base) + off; }

struct Stats {
  float *mu0, *r0, *mu1, *r1, *mu2, *r2, *muU, *rU, *muG, *rG;
};
Stats stats_of(const void* saved, const Layout& L, size_t N) {
  float* s = reinterpret_cast<float*>(const_cast<char*>(at(saved, L.stats)));
  Stats st;
  st.mu0 = s;
  st.r0 = s + N;
  st.mu1 = s + 2 * N;
  st.r1 = s + 3 * N;
  st.mu2 = s + 4 * N;
  st.r2 = s + 5 * N;
  st.muU = s + 6 * N;
  st.rU = s + 7 * N;
  st.muG = s + 8 * N;
  st.rG = s + 9 * N;
  return st;
}

// Samples [b0, b1) of chunk i of n (an even split of B).
inline int chunk_begin(int B, int i, int n) { return (int)((long long)B * i / n); }

// The forward over samples [b0, b1): every kernel of the forward works on
// whole rows (a sample's T rows for norm0 / token mix / norm1, single rows
// or per-token GEMM rows for the rest), so a range of samples is the same
// computation on a sub-batch at an offset of every [B, T, ...] buffer.
rmx_status forward_rows(const rmx_config& c, const Layout& L, const void* x, const rmx_params& p, void* saved,
                        void* y, cudaStream_t st, int b0, int b1) {
  const size_t N = (size_t)c.B * c.T;
  const size_t e = esize(c.dtype);
  const size_t r0 = (size_t)b0 * c.T;
  RowArgs ra = L.ra;
  ra.B = b1 - b0;
  if (ra.B <= 0) return RMX_OK;
  // Byte offsets of row r0 in buffers of D, H and 2H storage elements per row.
  const size_t oD = r0 * L.D * e, oH = r0 * L.H * e;
  void* out1 = at(saved, L.out1 + oD);
  void* Z = at(saved, L.Z + 2 * oH);
  void* hidden = at(saved, L.hidden + oH);
  void* s2 = at(saved, L.s2 + oD);
  void* s1 = at(saved, L.s1 + oD);
  const void* xr = at(x, oD);
  void* yr = at(y, oD);
  Stats S = stats_of(saved, L, N);
  for (float** v : {&S.mu0, &S.r0, &S.mu1, &S.r1, &S.mu2, &S.r2, &S.muU, &S.rU, &S.muG, &S.rG}) *v += r0;
  if (ln01_fwd_supported(ra)) {
    Launch l("ln01_fwd", st);
    RMX_TRY(l.done(launch_ln01_fwd(ra, xr, p.gamma0, p.beta0, p.gamma1, p.beta1, s1, out1, S.mu0, S.r0, S.mu1,
                                   S.r1, st)));
  } else {
    // Samples too large to stage: norm0 writes its output token-mixed into
    // the s1 buffer, norm1 adds x in place.
    {
      Launch l("ln0_fwd_mixed", st);
      RMX_TRY(l.done(launch_ln_fwd(ra, LNF_MIXED_OUT, xr, nullptr, p.gamma0, p.beta0, s1, S.mu0, S.r0, nullptr,
                                   st)));
    }
    {
      Launch l("ln1_fwd", st);
      RMX_TRY(l.done(launch_ln_fwd(ra, LNF_SUM_IN, s1, xr, p.gamma1, p.beta1, out1, S.mu1, S.r1, s1, st)));
    }
  }
  float* zstats = reinterpret_cast<float*>(at(saved, L.zstats)) + r0 * (size_t)zstats_tiles(L.H) * 4;
  const int sd = storage(c.dtype);
  const bool tf32 = c.dtype == RMX_F32_TF32;
  const int M = b1 - b0;
  // 16-bit rows up to H = 2560: the gate pass takes the statistics of Z
  // itself (row in registers) and GEMM1 stores Z with the bias alone;
  // otherwise GEMM1's epilogue (or a statistics pass) writes per-group
  // statistics of Z that the gate pass merges.
  const bool rows_gate = gate_fwd_rows_supported(ra);
  {
    GemmDesc d{tf32 ? GEMM_DGRAD : GEMM_FWD, rows_gate ? EPI_BIAS : EPI_BIAS_ZSTATS, sd, M, 2 * L.H, L.D, c.T,
               out1, tf32 ? at(saved, L.w1T) : p.w1, Z, p.b1, nullptr, rows_gate ? nullptr : zstats, L.H,
               tf32 ? 1 : 0};
    const bool epilogue_stats = !rows_gate && tc_engine(d);
    RMX_TRY(run_gemm("gemm1_fwd", d, st));
    if (!rows_gate && !epilogue_stats) {
      Launch l("zstats", st);
      RMX_TRY(l.done(launch_zstats(ra, Z, zstats, st)));
    }
  }
  {
    Launch l("gate_fwd", st);
    if (rows_gate)
      RMX_TRY(l.done(launch_gate_fwd_rows(ra, Z, S.muU, S.rU, S.muG, S.rG, p.lnx_w, p.lnx_b, p.lng_w, p.lng_b,
                                          hidden, st)));
    else
      RMX_TRY(l.done(launch_gate_fwd(ra, Z, zstats, S.muU, S.rU, S.muG, S.rG, p.lnx_w, p.lnx_b, p.lng_w,
                                     p.lng_b, hidden, st)));
  }
  {
    GemmDesc d{tf32 ? GEMM_DGRAD : GEMM_FWD, EPI_BIAS_RESID, sd, M, L.D, L.H, c.T, hidden,
               tf32 ? at(saved, L.woutT) : p.wout, s2, p.bout, out1, nullptr, 0, tf32 ? 1 : 0};
    RMX_TRY(run_gemm("gemm2_fwd", d, st));
  }
  {
    Launch l("ln2_fwd", st);
    RMX_TRY(l.done(launch_ln_fwd(ra, LNF_PLAIN, s2, nullptr, p.gamma2, p.beta2, yr, S.mu2, S.r2, nullptr, st)));
  }
  return RMX_OK;
}

// x_in (may be null): x arrives in kXChunks chunks of samples, event i
// recorded once chunk i is in device memory.  The forward then runs in
// kFwdChunks ranges of samples, each after the events of the x chunks it
// covers, so that its kernels overlap the rest of the upload (at the cost
// of reading the weights once per range).
rmx_status forward_impl(const rmx_config& c, const void* x, const rmx_params& p, void* saved, void* y,
                        cudaStream_t st, const cudaEvent_t* x_in = nullptr) {
  const Layout L = layout_of(c);
  // TF32: the weights as [T, N, K] (K-major) for the dgrad-form contraction.
  if (c.dtype == RMX_F32_TF32) {
    Launch l("tf32_transpose", st);
    RMX_TRY(l.done(launch_transpose_f32(static_cast<const float*>(p.w1), reinterpret_cast<float*>(at(saved, L.w1T)),
                                        c.T, L.D, 2 * L.H, (long long)L.D * 2 * L.H, 2 * L.H, L.D, st)));
    Launch l2("tf32_transpose", st);
    RMX_TRY(l2.done(launch_transpose_f32(static_cast<const float*>(p.wout),
                                         reinterpret_cast<float*>(at(saved, L.woutT)), c.T, L.H, L.D,
                                         (long long)L.H * L.D, L.D, L.H, st)));
  }
  const int n = x_in ? kFwdChunks : 1;
  for (int k = 0; k < n; ++k) {
    const int b0 = chunk_begin(c.B, k, n), b1 = chunk_begin(c.B, k + 1, n);
    if (x_in)
      for (int i = 0; i < kXChunks; ++i)
        if (chunk_begin(c.B, i, kXChunks) < b1 && chunk_begin(c.B, i + 1, kXChunks) > b0 &&
            cudaStreamWaitEvent(st, x_in[i], 0) != cudaSuccess)
          return RMX_ERR_CUDA;
    RMX_TRY(forward_rows(c, L, x, p, saved, y, st, b0, b1));
  }
  return RMX_OK;
}

// dx_ready (may be null) is recorded on `st` as soon as dx is final.
rmx_status backward_impl(const rmx_config& c, const void* x, const void* dy, const void* saved,
                         const rmx_params& p, void* dx, const rmx_grads& g, void* ws, cudaStream_t st,
                         cudaEvent_t dx_ready) {
  const Layout L = layout_of(c);
  const size_t N = (size_t)c.B * c.T;
  const void* out1 = at(saved, L.out1);
  const void* Z = at(saved, L.Z);
  const void* hidden = at(saved, L.hidden);
  const void* s2 = at(saved, L.s2);
  Stats S = stats_of(saved, L, N);
  void* ds2 = at(ws, L.ds2);
  void* dh = at(ws, L.dh);
  void* dZ = at(ws, L.dZ);
  void* dout1 = at(ws, L.dout1);
  void* ds1 = at(ws, L.ds1);
  void* da0 = at(ws, L.da0);
  const void* s1 = at(saved, L.s1);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(at(ws, off)); };
  const int sd = storage(c.dtype);
  const bool tf32 = c.dtype == RMX_F32_TF32;

  {
    Launch l("ln2_bwd", st);
    RMX_TRY(l.done(launch_ln2_bwd(L.ra, dy, s2, S.mu2, S.r2, p.gamma2, ds2, F(L.pg2), F(L.pb2), F(L.pbo), st)));
  }
  {
    GemmDesc d{GEMM_DGRAD, EPI_STORE, sd, c.B, L.H, L.D, c.T, ds2, p.wout, dh, nullptr, nullptr, nullptr, 0,
               tf32 ? 1 : 0};
    RMX_TRY(run_gemm("gemm2_dgrad", d, st));
  }
  {
    Launch l("gate_bwd", st);
    RMX_TRY(l.done(launch_gate_bwd(L.ra, dh, Z, S.muU, S.rU, S.muG, S.rG, p.lnx_w, p.lnx_b, p.lng_w, p.lng_b, dZ,
                                   F(L.pwx), F(L.pbx), F(L.pwg), F(L.pbg), F(L.pb1), st)));
  }
  {
    GemmDesc d{GEMM_DGRAD, EPI_RESID, sd, c.B, L.D, 2 * L.H, c.T, dZ, p.w1, dout1, nullptr, ds2, nullptr, 0,
               tf32 ? 1 : 0};
    RMX_TRY(run_gemm("gemm1_dgrad", d, st));
  }
  const bool gather0 = ln0_bwd_gather_supported(L.ra);
  if (gather0) {
    // norm1's backward writes ds1 alone; norm0's gathers its mixed-back
    // input from ds1 directly.
    {
      Launch l("ln1_bwd", st);
      RMX_TRY(l.done(launch_ln_bwd(L.ra, LNB_PLAIN, dout1, s1, S.mu1, S.r1, p.gamma1, nullptr, ds1, nullptr,
                                   F(L.pg1), F(L.pbe1), nullptr, st)));
    }
    {
      Launch l("ln0_bwd_gather", st);
      RMX_TRY(l.done(launch_ln0_bwd_gather(L.ra, ds1, x, S.mu0, S.r0, p.gamma0, dx, F(L.pg0), F(L.pb0), st)));
    }
  } else {
    {
      Launch l("ln1_bwd_mixed", st);
      RMX_TRY(l.done(launch_ln_bwd(L.ra, LNB_MIXED_TOO, dout1, s1, S.mu1, S.r1, p.gamma1, nullptr, ds1, da0,
                                   F(L.pg1), F(L.pbe1), nullptr, st)));
    }
    {
      Launch l("ln0_bwd", st);
      RMX_TRY(l.done(launch_ln_bwd(L.ra, LNB_RESID, da0, x, S.mu0, S.r0, p.gamma0, ds1, dx, nullptr,
                                   F(L.pg0), F(L.pb0), nullptr, st)));
    }
  }
  if (dx_ready && cudaEventRecord(dx_ready, st) != cudaSuccess) return RMX_ERR_CUDA;
  // Weight gradients last: every SM is busy with one GEMM CTA, so there is
  // nothing for a second stream to overlap them with.
  if (tf32) {
    // TF32: both operands K-major, the batch (padded to Bp with zeros) as K:
    // dW[t] = X[t] @ Y[t]^T with X = [T, M, Bp], Y = [T, N, Bp] transposed
    // copies, written as [T, M, N].
    auto tr = [&](const void* src, size_t off, int X) {
      Launch l("tf32_transpose", st);
      return l.done(launch_transpose_f32(static_cast<const float*>(src), reinterpret_cast<float*>(at(ws, off)),
                                         c.T, c.B, X, X, (long long)c.T * X, L.Bp, st));
    };
    RMX_TRY(tr(hidden, L.hT, L.H));
    RMX_TRY(tr(ds2, L.ds2T, L.D));
    RMX_TRY(tr(out1, L.out1T, L.D));
    RMX_TRY(tr(dZ, L.dZT, 2 * L.H));
    auto wgrad = [&](const char* name, int M, int N, size_t a, size_t b, void* out) {
      GemmDesc d{GEMM_DGRAD, EPI_STORE, sd, M, N, L.Bp, c.T, at(ws, a), at(ws, b), out, nullptr, nullptr, nullptr, 0, 1};
      d.a_gs = (long long)M * L.Bp;
      d.a_rs = L.Bp;
      d.c_gs = (long long)M * N;
      d.c_rs = N;
      return run_gemm(name, d, st);
    };
    RMX_TRY(wgrad("gemm2_wgrad", L.H, L.D, L.hT, L.ds2T, g.wout));
    RMX_TRY(wgrad("gemm1_wgrad", L.D, 2 * L.H, L.out1T, L.dZT, g.w1));
  } else {
    {
      GemmDesc d{GEMM_WGRAD, EPI_STORE, sd, L.H, L.D, c.B, c.T, hidden, ds2, g.wout, nullptr, nullptr};
      RMX_TRY(run_gemm("gemm2_wgrad", d, st));
    }
    {
      GemmDesc d{GEMM_WGRAD, EPI_STORE, sd, L.D, 2 * L.H, c.B, c.T, out1, dZ, g.w1, nullptr, nullptr};
      RMX_TRY(run_gemm("gemm1_wgrad", d, st));
    }
  }
  {
    ColsumJob jobs[kColsumJobs];
    colsum_jobs(L, c, &g, ws, jobs);
    Launch l("colsums", st);
    RMX_TRY(l.done(launch_colsums(jobs, kColsumJobs, sd, st)));
  }
  return RMX_OK;
}

// ------------------------------------------------------------------ padded blocks
const void* const* param_slots(const rmx_params& p) { return reinterpret_cast<const void* const*>(&p); }
void* const* grad_slots(const rmx_grads& g) { return reinterpret_cast<void* const*>(&g); }
static_assert(sizeof(rmx_params) == kNumParams * sizeof(void*), "14 parameter pointers");
static_assert(sizeof(rmx_grads) == kNumParams * sizeof(void*), "14 gradient pointers");

rmx_params params_at(void* base, const ParamSet& ps) {
  const void* v[kNumParams];
  for (int k = 0; k < kNumParams; ++k) v[k] = at(base, ps.off[k]);
  rmx_params p;
  std::memcpy(&p, v, sizeof(p));
  return p;
}
rmx_grads grads_at(void* base, const ParamSet& ps) {
  void* v[kNumParams];
  for (int k = 0; k < kNumParams; ++k) v[k] = at(base, ps.off[k]);
  rmx_grads g;
  std::memcpy(&g, v, sizeof(g));
  return g;
}

rmx_status pad_copy(const char* name, const void* src, void* dst, int dtype, const PadMap& m, bool pack,
                    cudaStream_t st) {
  Launch l(name, st);
  return l.done(launch_pad_copy(src, dst, dtype, m, pack, st));
}

// [B, T, D] activations between the caller's layout and the padded one.
PadMap act_map(const Layout& L, const rmx_config& c) {
  const int N = c.B * c.T;
  return PadMap{1, N, N, L.Dl, L.D, 1};
}

// Forward of a block whose rows need padding: x and the parameters are
// packed into `saved` (the backward reuses them), the padded block runs, and
// y is unpacked.
rmx_status forward_padded(const Layout& L, const rmx_config& c, const void* x, const rmx_params& p, void* saved,
                          void* y, cudaStream_t st) {
  RMX_TRY(pad_copy("pad_in", x, at(saved, L.xp), storage(c.dtype), act_map(L, c), true, st));
  const void* const* src = param_slots(p);
  for (int k = 0; k < kNumParams; ++k)
    RMX_TRY(pad_copy("pad_in", src[k], at(saved, L.pp.off[k]), storage(c.dtype), param_map(k, c.T, L.Dl, L.Hl, L.D, L.H),
                     true, st));
  RMX_TRY(forward_impl(c, at(saved, L.xp), params_at(saved, L.pp), saved, at(saved, L.yp), st));
  return pad_copy("pad_out", at(saved, L.yp), y, storage(c.dtype), act_map(L, c), false, st);
}

rmx_status backward_padded(const Layout& L, const rmx_config& c, const void* dy, const void* saved, void* dx,
                           const rmx_grads& g, void* ws, cudaStream_t st, cudaEvent_t dx_ready) {
  void* sv = const_cast<void*>(saved);
  RMX_TRY(pad_copy("pad_in", dy, at(ws, L.dyp), storage(c.dtype), act_map(L, c), true, st));
  const rmx_grads gp = grads_at(ws, L.gp);
  RMX_TRY(backward_impl(c, at(sv, L.xp), at(ws, L.dyp), saved, params_at(sv, L.pp), at(ws, L.dxp), gp, ws, st,
                        nullptr));
  RMX_TRY(pad_copy("pad_out", at(ws, L.dxp), dx, storage(c.dtype), act_map(L, c), false, st));
  if (dx_ready && cudaEventRecord(dx_ready, st) != cudaSuccess) return RMX_ERR_CUDA;
  void* const* dst = grad_slots(g);
  void* const* srcp = grad_slots(gp);
  for (int k = 0; k < kNumParams; ++k)
    RMX_TRY(pad_copy("pad_out", srcp[k], dst[k], storage(c.dtype), param_map(k, c.T, L.Dl, L.Hl, L.D, L.H), false, st));
  return RMX_OK;
}

rmx_status zero_grads(const rmx_config& c, const rmx_grads& g, cudaStream_t st) {
  const size_t e = esize(c.dtype), T = c.T, D = c.D, H = c.H;
  struct {
    void* p;
    size_t n;
  } z[] = {{g.w1, T * D * 2 * H}, {g.b1, T * 2 * H}, {g.wout, T * H * D}, {g.bout, T * D},
           {g.gamma0, D},         {g.beta0, D},      {g.gamma1, D},       {g.beta1, D},
           {g.gamma2, D},         {g.beta2, D},      {g.lnx_w, H},        {g.lnx_b, H},
           {g.lng_w, H},          {g.lng_b, H}};
  for (auto& q : z)
    if (cudaMemsetAsync(q.p, 0, q.n * e, st) != cudaSuccess) return RMX_ERR_CUDA;
  return RMX_OK;
}

// rmx_forward with x_in as in forward_impl (null: x is already there).
rmx_status forward_checked(const rmx_config* cfg, const void* x, const rmx_params* params, void* saved,
                           size_t saved_bytes, void* y, cudaStream_t st, const cudaEvent_t* x_in) {
  if (!config_ok(cfg)) return RMX_ERR_INVALID_ARG;
  RMX_TRY(check_params(params));
  if (cfg->B == 0) return RMX_OK;
  RMX_TRY(check_ptr(x));
  RMX_TRY(check_ptr(y));
  RMX_TRY(check_ptr(saved));
  if (x == y) return RMX_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  if (saved_bytes < L.saved_total) return RMX_ERR_WORKSPACE;
  RMX_TRY(kernels_support(*cfg));
  if (L.padded) {
    if (x_in)
      for (int i = 0; i < kXChunks; ++i)
        if (cudaStreamWaitEvent(st, x_in[i], 0) != cudaSuccess) return RMX_ERR_CUDA;
    return forward_padded(L, *cfg, x, *params, saved, y, st);
  }
  return forward_impl(*cfg, x, *params, saved, y, st, x_in);
}

rmx_status backward_checked(const rmx_config* cfg, const void* x, const void* dy, const void* saved,
                            size_t saved_bytes, const rmx_params* params, void* dx, const rmx_grads* grads,
                            void* ws, size_t ws_bytes, rmx_stream stream, cudaEvent_t dx_ready) {
  if (!config_ok(cfg)) return RMX_ERR_INVALID_ARG;
  RMX_TRY(check_params(params));
  RMX_TRY(check_grads(grads));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->B == 0) return zero_grads(*cfg, *grads, st);
  RMX_TRY(check_ptr(x));
  RMX_TRY(check_ptr(dy));
  RMX_TRY(check_ptr(saved));
  RMX_TRY(check_ptr(dx));
  RMX_TRY(check_ptr(ws));
  const Layout L = layout_of(*cfg);
  if (saved_bytes < L.saved_total || ws_bytes < L.ws_total) return RMX_ERR_WORKSPACE;
  RMX_TRY(kernels_support(*cfg));
  if (L.padded) return backward_padded(L, *cfg, dy, saved, dx, *grads, ws, st, dx_ready);
  return backward_impl(*cfg, x, dy, saved, *params, dx, *grads, ws, st, dx_ready);
}

}  // namespace
}  // namespace rmx

using namespace rmx;

extern "C" {

size_t rmx_saved_bytes(const rmx_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return layout_of(*cfg).saved_total;
}

size_t rmx_workspace_bytes(const rmx_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return layout_of(*cfg).ws_total;
}

rmx_status rmx_forward(const rmx_config* cfg, const void* x, const rmx_params* params, void* saved,
                       size_t saved_bytes, void* y, rmx_stream stream) {
  return forward_checked(cfg, x, params, saved, saved_bytes, y, reinterpret_cast<cudaStream_t>(stream), nullptr);
}



rmx_status rmx_backward(const rmx_config* cfg, const void* x, const void* dy, const void* saved,
                        size_t saved_bytes, const rmx_params* params, void* dx, const rmx_grads* grads,
                        void* ws, size_t ws_bytes, rmx_stream stream) {
  return backward_checked(cfg, x, dy, saved, saved_bytes, params, dx, grads, ws, ws_bytes, stream, nullptr);
}

rmx_status rmx_step_host(const rmx_config* cfg, const rmx_host_io* host, const rmx_device_io* dev,
                         const rmx_params* params, const rmx_grads* grads, void* saved, size_t saved_bytes,
                         void* ws, size_t ws_bytes, rmx_stream stream) {
  if (!config_ok(cfg) || !host || !dev) return RMX_ERR_INVALID_ARG;
  if (!host->x || !host->dy || !host->y || !host->dx) return RMX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)cfg->B * cfg->T * cfg->D * esize(cfg->dtype);
  if (cfg->B == 0) {
    RMX_TRY(rmx_forward(cfg, dev->x, params, saved, saved_bytes, dev->y, stream));
    return rmx_backward(cfg, dev->x, dev->dy, saved, saved_bytes, params, dev->dx, grads, ws, ws_bytes, stream);
  }
  RMX_TRY(check_ptr(dev->x));
  RMX_TRY(check_ptr(dev->dy));
  RMX_TRY(check_ptr(dev->y));
  RMX_TRY(check_ptr(dev->dx));
  // dy is not needed before the backward, y is final after the forward and
  // dx before the weight gradients: those copies run on the library's copy
  // stream, beside the compute, and are joined back to `stream` at the end.
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStream* cs = copy_stream();
  if (!cs) return RMX_ERR_CUDA;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // The copy stream must not overwrite dev->x or dev->dy while earlier work
  // on `stream` may read them.
  if (!ok(cudaEventRecord(cs->start, st)) || !ok(cudaStreamWaitEvent(cs->s, cs->start, 0))) return RMX_ERR_CUDA;
  // x in chunks of samples (the forward's first pass follows chunk by
  // chunk), then dy: one host->device engine serves them in that order.
  const size_t sample_bytes = (size_t)cfg->T * cfg->D * esize(cfg->dtype);
  for (int i = 0; i < kXChunks; ++i) {
    const size_t o = (size_t)chunk_begin(cfg->B, i, kXChunks) * sample_bytes;
    const size_t n = (size_t)chunk_begin(cfg->B, i + 1, kXChunks) * sample_bytes - o;
    if (n && !ok(cudaMemcpyAsync(static_cast<char*>(dev->x) + o, static_cast<const char*>(host->x) + o, n,
                                 cudaMemcpyHostToDevice, cs->s)))
      return RMX_ERR_CUDA;
    if (!ok(cudaEventRecord(cs->x_in[i], cs->s))) return RMX_ERR_CUDA;
  }
  if (!ok(cudaMemcpyAsync(dev->dy, host->dy, bytes, cudaMemcpyHostToDevice, cs->s))) return RMX_ERR_CUDA;
  if (!ok(cudaEventRecord(cs->dy_in, cs->s))) return RMX_ERR_CUDA;
  RMX_TRY(forward_checked(cfg, dev->x, params, saved, saved_bytes, dev->y, st, cs->x_in));
  if (!ok(cudaEventRecord(cs->fwd_done, st)) || !ok(cudaStreamWaitEvent(cs->s, cs->fwd_done, 0))) return RMX_ERR_CUDA;
  if (!ok(cudaMemcpyAsync(host->y, dev->y, bytes, cudaMemcpyDeviceToHost, cs->s))) return RMX_ERR_CUDA;
  if (!ok(cudaStreamWaitEvent(st, cs->dy_in, 0))) return RMX_ERR_CUDA;
  // dx is final before the weight gradients are computed: its download runs
  // beside them.
  RMX_TRY(backward_checked(cfg, dev->x, dev->dy, saved, saved_bytes, params, dev->dx, grads, ws, ws_bytes, stream,
                           cs->dx_ready));
  if (!ok(cudaStreamWaitEvent(cs->s, cs->dx_ready, 0))) return RMX_ERR_CUDA;
  if (!ok(cudaMemcpyAsync(host->dx, dev->dx, bytes, cudaMemcpyDeviceToHost, cs->s))) return RMX_ERR_CUDA;
  if (!ok(cudaEventRecord(cs->done, cs->s))) return RMX_ERR_CUDA;
  if (!ok(cudaStreamWaitEvent(st, cs->done, 0))) return RMX_ERR_CUDA;
  return RMX_OK;
}

// ------------------------------------------------------------------ graph replay
struct rmx_graph_st {
  cudaGraphExec_t exec = nullptr;
  long long launches = 0;  // kernel launches of one replay
};

rmx_status rmx_graph_create(const rmx_config* cfg, const void* x, const void* dy, const rmx_params* params,
                            void* saved, size_t saved_bytes, void* y, void* dx, const rmx_grads* grads, void* ws,
                            size_t ws_bytes, rmx_graph* out) {
  if (!out) return RMX_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg)) return RMX_ERR_INVALID_ARG;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return RMX_ERR_CUDA;
  // Relaxed capture: the first use of the library on a device looks up
  // symbol addresses and kernel attributes, which are not stream work.
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return RMX_ERR_CUDA;
  }
  const bool prof = g_prof.exchange(false);  // no profiling events inside a graph
  const long long l0 = g_launches.load();
  rmx_status st = rmx_forward(cfg, x, params, saved, saved_bytes, y, reinterpret_cast<rmx_stream>(cs));
  if (st == RMX_OK)
    st = rmx_backward(cfg, x, dy, saved, saved_bytes, params, dx, grads, ws, ws_bytes,
                      reinterpret_cast<rmx_stream>(cs));
  const long long n = g_launches.load() - l0;
  g_prof.store(prof);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (st != RMX_OK || ec != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return st != RMX_OK ? st : RMX_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return RMX_ERR_CUDA;
  rmx_graph g = new (std::nothrow) rmx_graph_st;
  if (!g) {
    cudaGraphExecDestroy(exec);
    return RMX_ERR_CUDA;
  }
  g->exec = exec;
  g->launches = n;
  *out = g;
  return RMX_OK;
}

rmx_status rmx_graph_launch(rmx_graph g, rmx_stream stream) {
  if (!g || !g->exec) return RMX_ERR_INVALID_ARG;
  if (cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RMX_ERR_CUDA;
  g_launches.fetch_add(g->launches);
  return RMX_OK;
}

rmx_status rmx_graph_destroy(rmx_graph g) {
  if (!g) return RMX_OK;
  const cudaError_t e = g->exec ? cudaGraphExecDestroy(g->exec) : cudaSuccess;
  delete g;
  return e == cudaSuccess ? RMX_OK : RMX_ERR_CUDA;
}

rmx_status rmx_check(rmx_stream stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RMX_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_rmx_error_word, sizeof(v)) != cudaSuccess) return RMX_ERR_CUDA;
  if (v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_rmx_error_word, &zero, sizeof(zero)) != cudaSuccess) return RMX_ERR_CUDA;
    return RMX_ERR_TIMEOUT;
  }
  return RMX_OK;
}

const char* rmx_status_str(rmx_status s) {
  switch (s) {
    case RMX_OK: return "RMX_OK";
    case RMX_ERR_INVALID_ARG: return "RMX_ERR_INVALID_ARG";
    case RMX_ERR_UNSUPPORTED: return "RMX_ERR_UNSUPPORTED";
    case RMX_ERR_ALIGNMENT: return "RMX_ERR_ALIGNMENT";
    case RMX_ERR_WORKSPACE: return "RMX_ERR_WORKSPACE";
    case RMX_ERR_CUDA: return "RMX_ERR_CUDA";
    case RMX_ERR_TIMEOUT: return "RMX_ERR_TIMEOUT";
  }
  return "RMX_ERR_UNKNOWN";
}

int rmx_version(void) { return 100; }

long long rmx_launch_count(void) { return g_launches.load(); }

rmx_status rmx_profile_enable(int on) {
  g_prof.store(on != 0);
  return RMX_OK;
}

rmx_status rmx_profile_select(const char* name) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_only = name ? name : "";
  return RMX_OK;
}

int rmx_profile_read(const char** names, long long* launches, double* total_ms, int cap) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    recs.swap(g_recs);
  }
  std::map<std::string, std::pair<long long, double>> agg;
  std::map<std::string, const char*> keep;
  std::vector<std::string> order;
  for (auto& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      std::string k(r.name);
      if (!agg.count(k)) {
        order.push_back(k);
        keep[k] = r.name;
      }
      agg[k].first += 1;
      agg[k].second += ms;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  int n = 0;
  for (auto& k : order) {
    if (n < cap && names && launches && total_ms) {
      names[n] = keep[k];
      launches[n] = agg[k].first;
      total_ms[n] = agg[k].second;
    }
    ++n;
  }
  return n;
}

rmx_status rmx_test_bounded_wait(int limit_us, rmx_stream stream) {
  if (limit_us <= 0 || limit_us > 10 * 1000 * 1000) return RMX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Launch l("bounded_wait_test", st);
  return l.done(launch_bounded_wait_test(device_error_word(), (unsigned long long)limit_us * 1000ull, st));
}

rmx_status rmx_test_gemm(int kind, int dtype, int M, int N, int K, int G, const void* A, const void* Bm, void* C,
                         rmx_stream stream) {
  if (kind < 0 || kind > 2 || dtype < 0 || dtype > 3) return RMX_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0) return RMX_ERR_INVALID_ARG;
  RMX_TRY(check_ptr(A));
  RMX_TRY(check_ptr(Bm));
  RMX_TRY(check_ptr(C));
  GemmDesc d{kind, EPI_STORE, storage(dtype), M, N, K, G, A, Bm, C, nullptr, nullptr, nullptr, 0,
             dtype == RMX_F32_TF32 ? 1 : 0};
  return run_gemm("test_gemm", d, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
