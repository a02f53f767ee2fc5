// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace rmx {

// ------------------------------------------------------------------ row passes
// D and H are the row pitches of the tensors the kernels see (multiples of
// 8); Dl and Hl the block's own sizes (Dl <= D, Hl <= H).  When they differ,
// every tensor is a zero-padded copy: columns Dl .. D-1 (and, for Z = [U | G]
// of pitch 2H, columns Hl .. H-1 of each half) hold zeros on input, means and
// variances are taken over the Dl (Hl) real columns, and the kernels write
// zeros there on output.
struct RowArgs {
  int B, T, D, H, dtype;
  int Dl, Hl;    // logical row lengths
  int nb;        // samples per CTA in the per-token gate backward
  int nbblk;     // ceil(B / nb)
  int nb_ln;     // samples per CTA in the LayerNorm backward
  int nbblk_ln;  // ceil(B / nb_ln)
};

// LayerNorm forward, one row per warp.  Modes: plain; output written
// token-mixed (column i*C+c of row j lands in row i, column j*C+c of the same
// sample, C = D/T); input is the sum of two tensors.
// LNF_SUM_IN rounds s + s_add to the storage type, normalises those values
// and also writes them to s_out (which may be s itself).
enum LnFwdMode { LNF_PLAIN = 0, LNF_MIXED_OUT = 1, LNF_SUM_IN = 2 };
cudaError_t launch_ln_fwd(const RowArgs& a, int mode, const void* s, const void* s_add, const void* g,
                          const void* be, void* y, float* mu, float* rs, void* s_out, cudaStream_t st);
// norm0 -> token mix -> + x -> norm1: writes s1 (norm1's input, rounded to
// the storage type), out1 and both row statistics.  With T a multiple of 8
// (up to 64) a cluster of T/8 CTAs per sample, each staging its 8 rows and
// the column stripe of the sample they need; otherwise one CTA per sample
// staging all its rows.  Supported when that fits in shared memory.
bool ln01_fwd_supported(const RowArgs& a);
cudaError_t launch_ln01_fwd(const RowArgs& a, const void* x, const void* gamma0, const void* beta0,
                            const void* gamma1, const void* beta1, void* s1, void* out1, float* mu0, float* r0,
                            float* mu1, float* r1, cudaStream_t st);
// LayerNorm backward over CTAs (t, b-block) of up to nb_ln <= kLnBwdMaxRows
// rows; per-CTA partial sums of dgamma and dbeta ([nbblk_ln*T][D]).  Modes:
// LNB_BIAS also sums ds per token into pbias; LNB_MIXED_TOO also writes
// token_mix(ds) to out_mixed; LNB_RESID adds resid to the output.
// LNB_PLAIN writes only the gradient.
constexpr int kLnBwdMaxRows = 64;
// CTAs of the LayerNorm backward ring resident per SM (occupancy of the
// launch shape with kLnBwdMaxRows rows), for choosing nb_ln.
int ln_bwd_ctas_per_sm(const RowArgs& a);
enum LnBwdMode { LNB_BIAS = 0, LNB_MIXED_TOO = 1, LNB_RESID = 2, LNB_PLAIN = 3 };
cudaError_t launch_ln_bwd(const RowArgs& a, int mode, const void* gin, const void* s,
                          const float* mu, const float* rs, const void* gamma, const void* resid, void* out,
                          void* out_mixed, float* pg, float* pb, float* pbias, cudaStream_t st);
// Backward of norm0 from ds1 (the gradient at norm1's input) without a
// token-mixed intermediate: dx = ds1 + LN0_backward(da0) with da0 = ds1 mixed
// back, gathered from a column stripe of ds1 staged in shared memory.  A CTA
// owns 8 rows of kLn0SamplesPerCta consecutive samples; partial sums of
// dgamma0 and dbeta0 go to [ln0_bwd_partial_rows][D].  Supported when
// T % 8 == 0 and a row is at most 160 16-byte vectors.
constexpr int kLn0SamplesPerCta = 4;
int ln0_bwd_partial_rows(const RowArgs& a);
bool ln0_bwd_gather_supported(const RowArgs& a);
cudaError_t launch_ln0_bwd_gather(const RowArgs& a, const void* ds1, const void* x, const float* mu0,
                                  const float* r0, const void* gamma0, void* dx, float* pg0, float* pb0,
                                  cudaStream_t st);
// Backward of norm2 (launch_ln_bwd in LNB_BIAS mode): ds2 plus partial sums
// for gamma2, beta2 and bout.
cudaError_t launch_ln2_bwd(const RowArgs& a, const void* dy, const void* s2, const float* mu2,
                           const float* r2, const void* g2, void* ds2, float* pg2, float* pb2,
                           float* pbo, cudaStream_t st);
// Forward of the gate, one pass: the per-row mean and 1/sqrt(var+eps) of U
// and G merged from `zstats` (see below) and written to muU, rU, muG, rG;
// then hidden = LN_x(U) * silu(LN_gate(G)) from Z = [U | G].
cudaError_t launch_gate_fwd(const RowArgs& a, const void* Z, const float* zstats, float* muU, float* rU,
                            float* muG, float* rG, const void* wx, const void* bx, const void* wg, const void* bg,
                            void* hidden, cudaStream_t st);
// The same with the statistics taken in-pass from the row held in
// registers (16-bit storage, H <= 2560): Z needs no group statistics.
bool gate_fwd_rows_supported(const RowArgs& a);
cudaError_t launch_gate_fwd_rows(const RowArgs& a, const void* Z, float* muU, float* rU, float* muG, float* rG,
                                 const void* wx, const void* bx, const void* wg, const void* bg, void* hidden,
                                 cudaStream_t st);
// Single-pass gate backward: dZ and the column partials of lnx_w, lnx_b,
// lng_w, lng_b ([nbblk*T, H] each) and b1 ([nbblk, T, 2H]) from dh, Z and the
// forward's inner-LayerNorm statistics.  CTA (bblk, t) owns up to nb <=
// kGateBwdMaxRows rows of token t and the whole row.
constexpr int kGateBwdMaxRows = 256;
int gate_bwd_ctas_per_sm(const RowArgs& a);
bool gate_bwd_fused_supported(const RowArgs& a);
cudaError_t launch_gate_bwd(const RowArgs& a, const void* dh, const void* Z, const float* muU, const float* rU,
                            const float* muG, const float* rG, const void* wx, const void* bx, const void* wg,
                            const void* bg, void* dZ, float* pwx, float* pbx, float* pwg, float* pbg, float* pb1,
                            cudaStream_t st);

// Deterministic column sums: out[j] = sum_{p<P} part[p*J + j], cast to dtype.
struct ColsumJob {
  const float* part;
  void* out;
  int P, J;
};
// One launch; the summation order is fixed (the same bits on every call).
constexpr int kMaxColsumJobs = 12;
cudaError_t launch_colsums(const ColsumJob* jobs, int njobs, int dtype, cudaStream_t st);

// Largest thread count a row pass may use (one thread per 16-byte vector).
constexpr int kRowThreadsMax = 512;
int max_dynamic_smem_bytes();

// ------------------------------------------------------------------ padding
// Gathers between a tensor of logical shape [outer][rows][cols] (row-major)
// and its zero-padded copy [outer][rows_p][cols_p]: the columns are split
// into `halves` equal parts, part h landing at column h * cols_p / halves of
// the padded row.  pack: padded <- logical (zeros in every padded place);
// unpack: logical <- padded.  Element type by dtype (0 f32, 1 bf16, 2 f16).
struct PadMap {
  int outer, rows, rows_p, cols, cols_p, halves;
};
cudaError_t launch_pad_copy(const void* src, void* dst, int dtype, const PadMap& m, bool pack, cudaStream_t st);
// Batched fp32 transpose for the TF32 contractions, whose operands must be
// K-major: dst[g][c][r] = src[g*gs + r*rs + c] (r < R), zero for R <= r < Rp.
cudaError_t launch_transpose_f32(const float* src, float* dst, int G, int R, int Cc, long long gs, long long rs,
                                 int Rp, cudaStream_t st);

// ------------------------------------------------------------------ GEMMs
enum GemmKind { GEMM_FWD = 0, GEMM_DGRAD = 1, GEMM_WGRAD = 2 };
enum GemmEpi {
  EPI_STORE = 0,
  EPI_BIAS = 1,
  EPI_BIAS_RESID = 2,
  EPI_RESID = 3,
  EPI_BIAS_ZSTATS = 4,    // + per-group statistics of Z (GEMM1 forward)
};

// Row statistics of Z = [U | G] in 128-column groups: for row r and group j
// (columns [128 j, 128 j + 128) of the 2H-wide row), zstats[(r * groups + j)
// * 4 + {0,1,2,3}] = {mean, M2} of the group's U columns and {mean, M2} of its
// G columns, taken from the stored (rounded) Z values.  M2 = sum of squared
// deviations from the mean.  Written by the GEMM1 epilogue (EPI_BIAS_ZSTATS)
// or by launch_zstats; merged per row by the gate forward.
constexpr int kZStatsTile = 128;
__host__ __device__ inline int zstats_tiles(int H) { return (2 * H + kZStatsTile - 1) / kZStatsTile; }
cudaError_t launch_zstats(const RowArgs& a, const void* Z, float* zstats, cudaStream_t st);

// One grouped GEMM over G groups (the tokens t).  Layouts, all row-major:
//   FWD:   C[m,g,:] = A[m,g,:] @ Bm[g]        A [M,G,K], Bm [G,K,N], C [M,G,N]
//   DGRAD: C[m,g,:] = A[m,g,:] @ Bm[g]^T      A [M,G,K], Bm [G,N,K], C [M,G,N]
//   WGRAD: C[g]     = A[:,g,:]^T @ Bm[:,g,:]  A [K,G,M], Bm [K,G,N], C [G,M,N]
// Epilogue: + bias[g,n] (bias [G,N]) and/or + resid (same layout as C).
struct GemmDesc {
  int kind, epi, dtype;
  int M, N, K, G;
  const void* A;
  const void* Bm;
  void* C;
  const void* bias;
  const void* resid;
  float* zstats;  // EPI_BIAS_ZSTATS only
  int split;      // EPI_BIAS_ZSTATS: first column of the G half (H)
  // fp32 (dtype 0): 1 runs the contraction on the tensor cores with TF32
  // operands (dgrad form only; see gemm_tc_supported), 0 on the CUDA cores.
  int tf32 = 0;
  // Optional element strides of A's (g, m) and C's (g, m) indices in the
  // FWD / DGRAD forms (0: the [M, G, K] / [M, G, N] defaults); TF32 only.
  long long a_gs = 0, a_rs = 0, c_gs = 0, c_rs = 0;
};

bool gemm_tc_supported(const GemmDesc& d);
cudaError_t gemm_tc_launch(const GemmDesc& d, unsigned int* err, cudaStream_t st);
cudaError_t gemm_simt_launch(const GemmDesc& d, cudaStream_t st);

// Test hook: a kernel that waits on an mbarrier nothing completes.
cudaError_t launch_bounded_wait_test(unsigned int* err, unsigned long long limit_ns, cudaStream_t st);

int sm_count();

// Rank-2 tiled tensor map without swizzle over a row-major [d1][d0] array of
// the storage dtype (0 f32, 1 bf16, 2 f16), row stride s1 bytes, box
// {b0, b1}; out-of-range elements of a box read as zero.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int dtype, uint64_t d0, uint64_t d1, uint64_t s1,
                        uint32_t b0, uint32_t b1);

}  // namespace rmx
