// Grouped GEMM on Blackwell tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Computes the four per-token contractions of the RankMixer block (page
// "Subgraph-fusion-based Mega-kernel Generation", section "Exact
// computation": Z[b,t] = out1[b,t] @ w1[t] + b1[t] and out2[b,t] =
// hidden[b,t] @ wout[t] + bout[t]) and the dgrad / wgrad contractions of
// their backward, for 16-bit storage (bf16 or fp16) with fp32 accumulation.
//
// Design (one CTA per SM, persistent over tiles):
//   warp 0     TMA producer: loads each k-block's A and B slices into a
//              shared-memory ring (128-byte swizzle): six stages of 32 KB
//              for a CTA pair, four of 48 KB for a CTA alone; the `full`
//              mbarriers count the bytes;
//   warp 1     allocates 512 TMEM columns; one thread issues tcgen05.mma
//              (kind::f16, K=16); each stage goes back to the producer by
//              tcgen05.commit on its `empty` barrier; the accumulator
//              alternates between two 256-column TMEM halves so the epilogue
//              of tile i overlaps the main loop of tile i+1;
//   warps 2-9  epilogue: two warps per TMEM lane quarter, each draining half
//              of the tile's columns 64 at a time (tcgen05.ld), releasing the
//              accumulator after its last load, applying bias / residual /
//              Z statistics in fp32 and writing 32x64 boxes through a
//              swizzled staging buffer with TMA stores.
// Paired mode (M spans at least two 128-row tiles): a cluster of two CTAs
// owns a 256x256 output tile.  The even CTA issues
// tcgen05.mma.cta_group::2 (M=256, N=256) over A split by rows and B split by
// columns between the two CTAs' shared memory; the odd CTA's copies count
// their bytes on the even CTA's `full` barrier, and the even CTA's commits
// are multicast to both CTAs' barriers.
// Operands are addressed through tensor maps so that per-token slices of
// [B,T,X] activations and [T,X,Y] weights need no copies; K-major and
// MN-major shared-memory layouts cover the NN (forward), NT (dgrad) and TN
// (wgrad) cases without transposes.  An MN-major operand whose MN extent is a
// multiple of 64 comes through a rank-5 map that stages the 1 KB swizzle
// atoms of one K group next to each other (see Params::mn_il).  TMA zero-fills
// out-of-range rows and columns, so ragged M, N and K need no special path.
//
// Every mbarrier wait is bounded (common.cuh); on expiry the kernel records
// an error bit, drains what it has in flight and frees its TMEM.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace rmx {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;  // BK, UMMA_K: 16-bit elements
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_BYTES = BN * BK * 2;           // 32 KB
constexpr int MN_CHUNK_BYTES = BK * 128;       // one 64-wide MN chunk of an MN-major tile
// A k-block is one 128-byte swizzle row of every operand row: 64 elements of
// a 16-bit type, 32 of fp32 (read by the tensor cores as TF32); one MMA
// takes 32 bytes of K (16 or 8 elements), four per k-block either way.
template <typename T> struct KBlock {
  static constexpr int E = 128 / (int)sizeof(T);
  static constexpr int MMA_K = 32 / (int)sizeof(T);
};
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = NUM_ACC * BN;        // 512
constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter
constexpr int THREADS = 64 + 32 * EPI_WARPS;   // producer, MMA, epilogue

// Shared-memory ring.  Single CTA: the whole 256-row B tile per stage, four
// stages.  CTA pair: each CTA holds its 128 rows of A and its half of B, so a
// stage is 32 KB and six fit.
template <bool PAIR> struct Ring {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int B_STAGE = PAIR ? B_BYTES / 2 : B_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_STAGE;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NUM_ACC + 1;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_WARPS * 4096 + 256;
  static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");
};
constexpr uint64_t kDrainLimitNs = 50ull * 1000ull * 1000ull;

struct Params {
  int M, N, K, G;
  int tiles_m, tiles_n, tiles_per_group, num_tiles, num_kb;
  int pairs_m, pair_tiles_per_group, num_pair_tiles;  // paired mode
  void* out;
  long long out_rs, out_gs;
  const void* bias;
  long long bias_gs;
  const void* resid;
  long long res_rs, res_gs;
  unsigned int* err;
  unsigned long long wait_limit_ns;
  float* zstats;  // EPI_BIAS_ZSTATS
  int split, zgroups;
  // 1: the MN-major operands come through rank-5 maps that lay a stage out as
  // [K group of 8][64-wide MN chunk][8 K rows][64 MN] (swizzle atoms of the
  // chunks of one K group adjacent), one TMA copy per operand and stage.
  int mn_il;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Same copy for a CTA pair: the data lands in this CTA's shared memory and
// the byte count is signalled on `bar`, which may be the peer CTA's barrier
// (a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Rank-5 forms of the two copies above (the interleaved MN-major operands).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// shared::cluster address of the variable at `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on a barrier that may live in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait_bounded with cluster-scope acquire (the arrivals come from the
// peer CTA as well).
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                          unsigned int* err, unsigned int errbit,
                                                          volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (((++n) & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(err, errbit);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Prefetch of the 128-byte line holding p into L1 (a hint; no fault on any
// address this kernel could read).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// TMEM allocation.  For a CTA pair (cta_group::2) one warp of each CTA
// executes these together.
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  if (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T: kind::f16 (fp16 or bf16 in) or, for
// fp32 operands, kind::tf32; fp32 accumulation.  For a CTA pair (issued by
// the even CTA only) A and D are split by rows and B by columns between the
// two CTAs, at the same shared / TMEM offsets.
template <typename T, bool PAIR>
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
  if (std::is_same<T, float>::value) {
    if (PAIR)
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "setp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
          ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "setp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
          ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
          : "memory");
    return;
  }
  if (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
template <bool PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// Pair: arrive on the barrier at `bar`'s offset in both CTAs once the
// tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}
// 32 lanes x 64 consecutive fp32 columns; thread i of the warp gets lane
// (quarter base + i).  The wait is in the same statement so that no use of
// the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld_32x64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled tile:
// start address, leading-dimension byte offset, stride-dimension byte offset
// (all >> 4), the fixed descriptor version bit (46) and the swizzle mode
// (bits 61-63: 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor, kind::f16 / kind::tf32: D fp32 (bits 4-5 = 1),
// A/B type (bits 7-9 / 10-12: 0 = fp16, 1 = bf16, 2 = tf32), A/B major
// (bits 15 / 16: 0 = K-major, 1 = MN-major), N >> 3 (bits 17-22), M >> 4
// (bits 24-28).
template <typename T, bool A_MN, bool B_MN, int UMMA_M>
__host__ __device__ constexpr uint32_t make_idesc() {
  constexpr uint32_t ab = std::is_same<T, bf16>::value ? 1u : std::is_same<T, float>::value ? 2u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(UMMA_M >> 4) << 24);
}

template <int KIND> struct KindTraits;
// forward:  A = activation [M,G,K] K-major; B = weight [G,K,N] MN-major
template <> struct KindTraits<GEMM_FWD> { static constexpr bool A_MN = false, B_MN = true, B_ACT = false; };
// dgrad:    A = activation [M,G,K] K-major; B = weight [G,N,K] K-major
template <> struct KindTraits<GEMM_DGRAD> { static constexpr bool A_MN = false, B_MN = false, B_ACT = false; };
// wgrad:    A = activation [K,G,M] MN-major; B = activation [K,G,N] MN-major
template <> struct KindTraits<GEMM_WGRAD> { static constexpr bool A_MN = true, B_MN = true, B_ACT = true; };

__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& g, int& m0, int& n0) {
  g = tile / p.tiles_per_group;
  const int rem = tile - g * p.tiles_per_group;
  const int tn = rem / p.tiles_m;
  const int tm = rem - tn * p.tiles_m;
  m0 = tm * BM;
  n0 = tn * BN;
}

// Paired mode: pair tile -> (group, this CTA's m0, n0).
__device__ __forceinline__ void pair_tile_coords(const Params& p, int pt, int rank, int& g, int& m0, int& n0) {
  g = pt / p.pair_tiles_per_group;
  const int rem = pt - g * p.pair_tiles_per_group;
  const int tn = rem / p.pairs_m;
  const int tp = rem - tn * p.pairs_m;
  m0 = (2 * tp + rank) * BM;
  n0 = tn * BN;
}

// Shifted sums of one half of a Z row over one column group, kept as pairs
// (even and odd columns) for the packed fp32x2 arithmetic.
struct ZSums {
  float n, k;   // count, shift
  float2 s, q;  // sum(x - k), sum((x - k)^2)
};

// Two floats rounded to the storage type, packed into 32 bits (lower
// column in the low half).
template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<bf16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<f16>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// The stored values of a packed word, back as floats (exact).
template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<bf16>(uint32_t w) { return bf16x2_to_f2(w); }
template <> __device__ __forceinline__ float2 unpack2<f16>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Epilogue of 32 consecutive columns n_base .. n_base+31 of row m: bias /
// residual in fp32, the Z statistics, and the result rounded and packed into
// pk[0..15] (16-bit output, two columns per word) or pk[0..31] (fp32 output).
// Columns at or past N (and rows past M) are computed from whatever the
// accumulator holds; the tensor store clips them.
template <typename T, int EPI>
__device__ __forceinline__ void epilogue_convert(const Params& p, int g, int m, int n_base, const float* v,
                                                 ZSums* zs, uint32_t* pk) {
  constexpr int V = VecN<T>::value;
#pragma unroll
  for (int c = 0; c < 32; c += V) {
    const int n = n_base + c;
    float o[V];
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] = v[c + e];
    const bool in = n < p.N && m < p.M;
    if (in) {
      if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_ZSTATS) {
        float bv[V];
        load_vec(reinterpret_cast<const T*>(p.bias) + (size_t)g * p.bias_gs + n, bv);
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] += bv[e];
      }
      if (EPI == EPI_RESID || EPI == EPI_BIAS_RESID) {
        float rv[V];
        load_vec(reinterpret_cast<const T*>(p.resid) + (size_t)g * p.res_gs + (size_t)m * p.res_rs + n, rv);
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] += rv[e];
      }
    }
    if constexpr (sizeof(T) == 4) {
#pragma unroll
      for (int e = 0; e < V; ++e) pk[c + e] = __float_as_uint(o[e]);
    } else {
#pragma unroll
      for (int e = 0; e < V; e += 2) pk[(c + e) >> 1] = pack2<T>(o[e], o[e + 1]);
    }
    if (EPI == EPI_BIAS_ZSTATS && in) {
      // Shifted sums of the stored (rounded) values of this half, read back
      // from the words just packed: the shift is the half's first value in
      // this column group, so the centred second moment is formed without
      // cancellation trouble.
      float2 r[V / 2];
#pragma unroll
      for (int e = 0; e < V; e += 2) {
        if constexpr (sizeof(T) == 4) r[e / 2] = make_float2(o[e], o[e + 1]);
        else r[e / 2] = unpack2<T>(pk[(c + e) >> 1]);
      }
      // Constant indices only, so the sums stay in registers.
      auto add = [&](ZSums& z) {
        if (z.n == 0.f) z.k = r[0].x;
        const float2 nk = f2(-z.k);
#pragma unroll
        for (int e = 0; e < V / 2; ++e) {
          const float2 dv = add2(r[e], nk);
          z.s = add2(z.s, dv);
          z.q = fma2(dv, dv, z.q);
        }
        z.n += (float)V;
      };
      if (n < p.split) add(zs[0]);
      else add(zs[1]);
    }
  }
}

// Tensor store of a shared-memory box (bulk async group).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the shared memory of every committed store has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <typename T, int KIND, int EPI, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const Params p) {
  // Setup (barriers, TMEM, tensor-map prefetch) overlaps the previous
  // kernel's tail; global memory is touched only after pdl_wait().
  pdl_trigger();
  using KT = KindTraits<KIND>;
  using R = Ring<PAIR>;
  constexpr int STAGES = R::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  // Output staging: one 32-row x 64-column box (4 KB, 128-byte swizzle) per
  // epilogue warp, after the ring (1024-byte aligned).
  const uint32_t sStage = sA + STAGES * R::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * R::STAGE_BYTES + EPI_WARPS * 4096);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + R::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + NUM_ACC + a); };
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 2 * NUM_ACC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_rank() : 0;
  // Work list: single tiles (this CTA), or pair tiles (this cluster).
  const int first = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int stride = PAIR ? (int)num_clusters_x() : (int)gridDim.x;
  const int count = PAIR ? p.num_pair_tiles : p.num_tiles;
  auto coords = [&](int it, int r, int& g, int& m0, int& n0) {
    if (PAIR) pair_tile_coords(p, it, r, g, m0, n0);
    else tile_coords(p, it, g, m0, n0);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);    // the (even) CTA's expect_tx arrival
      mbar_init(empty_bar(s), 1);   // one MMA commit per use
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      // One arrive per epilogue warp, of both CTAs for a pair.
      mbar_init(tempty_bar(a), PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_map(&tmA);
    prefetch_map(&tmB);
    prefetch_map(&tmC);
  }
  if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // Pair: the peer's barriers are initialised before anything is signalled
  // on them.
  if (PAIR) cluster_barrier();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = first; ok && tile < count; tile += stride) {
        // Pieces of the tile that CTA r requests.  MN-major tiles come as
        // 64-wide chunks; chunks or tiles wholly past M or N are skipped
        // (they only feed discarded outputs) and not counted.
        auto a_pieces = [&](int m0) {
          return KT::A_MN ? max(0, min(BM / 64, (p.M - m0 + 63) / 64)) : (m0 < p.M ? 1 : 0);
        };
        // B columns [nb0, nb0 + nw) held by CTA r: the whole tile alone, half
        // of it in a pair.
        auto b_pieces = [&](int nb0, int nw) {
          return KT::B_MN ? max(0, min(nw / 64, (p.N - nb0 + 63) / 64)) : (nb0 < p.N ? 1 : 0);
        };
        constexpr int B_W = PAIR ? BN / 2 : BN;
        int g, m0, n0;
        coords(tile, rank, g, m0, n0);
        const int nb0 = n0 + (PAIR ? rank * B_W : 0);
        const int a_n = a_pieces(m0), b_n = b_pieces(nb0, B_W);
        const uint32_t a_piece = KT::A_MN ? MN_CHUNK_BYTES : A_BYTES;
        const uint32_t b_piece = KT::B_MN ? MN_CHUNK_BYTES : R::B_STAGE;
        // Bytes of `n` requested pieces: an interleaved MN-major operand comes
        // as one box of the whole stage (its chunks past M or N zero-filled).
        auto a_bytes = [&](int n) { return (KT::A_MN && p.mn_il) ? (n > 0 ? (uint32_t)A_BYTES : 0u) : n * a_piece; };
        auto b_bytes = [&](int n) {
          return (KT::B_MN && p.mn_il) ? (n > 0 ? (uint32_t)R::B_STAGE : 0u) : n * b_piece;
        };
        // The even CTA's full barrier counts the bytes of both CTAs.
        uint32_t tx = a_bytes(a_n) + b_bytes(b_n);
        if (PAIR) {
          int g1, m1, n1;
          coords(tile, 1, g1, m1, n1);
          tx += a_bytes(a_pieces(m1)) + b_bytes(b_pieces(n0 + B_W, B_W));
        }
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, p.wait_limit_ns, p.err, ERRBIT_WAIT_PRODUCER,
                                 abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = PAIR ? mapa_shared(full_bar(s), 0) : full_bar(s);
          if (rank == 0) mbar_expect_tx(full_bar(s), tx);
          auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
            if (PAIR) tma_load_3d_pair(dst, map, fb, c0, c1, c2);
            else tma_load_3d(dst, map, fb, c0, c1, c2);
          };
          auto load5 = [&](uint32_t dst, const CUtensorMap* map, int mn, int k, int gg) {
            // map {64, 8, MN / 64, K / 8, G}: whole stage from chunk mn / 64, K group k / 8
            if (PAIR) tma_load_5d_pair(dst, map, fb, 0, 0, mn / 64, k / 8, gg);
            else tma_load_5d(dst, map, fb, 0, 0, mn / 64, k / 8, gg);
          };
          const int k0 = kb * KBlock<T>::E;
          const uint32_t a_dst = sA + s * A_BYTES, b_dst = sB + s * R::B_STAGE;
          if (!KT::A_MN) {
            if (a_n) load(a_dst, &tmA, k0, g, m0);                                      // map {K, G, M}
          } else if (p.mn_il) {
            if (a_n) load5(a_dst, &tmA, m0, k0, g);
          } else {
            for (int c = 0; c < a_n; ++c) load(a_dst + c * MN_CHUNK_BYTES, &tmA, m0 + 64 * c, g, k0);  // {M, G, K}
          }
          if (!KT::B_MN) {
            if (b_n) load(b_dst, &tmB, k0, nb0, g);                                     // map {K, N, G}
          } else if (p.mn_il) {
            if (b_n) load5(b_dst, &tmB, nb0, k0, g);
          } else {
            for (int c = 0; c < b_n; ++c) {
              if (!KT::B_ACT) load(b_dst + c * MN_CHUNK_BYTES, &tmB, nb0 + 64 * c, k0, g);  // map {N, K, G}
              else load(b_dst + c * MN_CHUNK_BYTES, &tmB, nb0 + 64 * c, g, k0);            // map {N, G, K}
            }
          }
        }
      }
      if (ok) {
        // Wait until the MMAs have released the last stages, so that no
        // commit is still on its way to this CTA's barriers at the end.
        const int first_j = it > STAGES ? it - STAGES : 0;
        for (int j = first_j; j < it; ++j)
          mbar_wait_bounded(empty_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, p.wait_limit_ns, p.err,
                            ERRBIT_WAIT_DRAIN, abort_flag);
      } else if (!PAIR || rank == 0) {
        // Let the copies already issued land before the CTA can exit.  A
        // pair's full barriers live in the even CTA and count the bytes of
        // both CTAs, so the even CTA's drain also covers the odd CTA's copies
        // of every stage it had armed; the pair's final cluster barrier keeps
        // the odd CTA alive until then.
        const int first_j = it > STAGES ? it - STAGES : 0;
        for (int j = first_j; j < it; ++j) {
          volatile int no_abort = 0;
          mbar_wait_bounded(full_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, kDrainLimitNs, p.err,
                            ERRBIT_WAIT_DRAIN, &no_abort);
        }
      } else {
        // The odd CTA of a pair has no barrier of its own to wait on: copies
        // of a stage the even CTA never armed get a fixed, ample time to land.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc<T, KT::A_MN, KT::B_MN, PAIR ? 2 * BM : BM>();
      int it = 0, lt = 0;
      bool ok = true;
      for (int tile = first; ok && tile < count; tile += stride, ++lt) {
        const int acc = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        const bool got = PAIR ? mbar_wait_bounded_cluster(tempty_bar(acc), aph ^ 1u, p.wait_limit_ns, p.err,
                                                          ERRBIT_WAIT_MMA, abort_flag)
                              : mbar_wait_bounded(tempty_bar(acc), aph ^ 1u, p.wait_limit_ns, p.err,
                                                  ERRBIT_WAIT_MMA, abort_flag);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(full_bar(s), ph, p.wait_limit_ns, p.err, ERRBIT_WAIT_MMA, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = sA + s * A_BYTES, b_base = sB + s * R::B_STAGE;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // K-major: advance 16 elements (32 bytes) inside the swizzle atom.
            // MN-major by chunks: advance 16 rows of 128 bytes; MN atoms one
            // chunk apart, K groups 1 KB apart.  Interleaved MN-major: advance
            // two K groups; MN atoms 1 KB apart, K groups (chunks x 1 KB) apart.
            constexpr uint32_t A_CH = BM / 64, B_CH = (PAIR ? BN / 2 : BN) / 64;
            const uint64_t adesc =
                KT::A_MN ? (p.mn_il ? sw128_desc(a_base + k * 2 * A_CH * 1024, 1024, A_CH * 1024)
                                    : sw128_desc(a_base + k * 2048, MN_CHUNK_BYTES, 1024))
                         : sw128_desc(a_base + k * 32, 16, 1024);
            const uint64_t bdesc =
                KT::B_MN ? (p.mn_il ? sw128_desc(b_base + k * 2 * B_CH * 1024, 1024, B_CH * 1024)
                                    : sw128_desc(b_base + k * 2048, MN_CHUNK_BYTES, 1024))
                         : sw128_desc(b_base + k * 32, 16, 1024);
            umma<T, PAIR>(d_tmem, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          if (PAIR) umma_commit_pair(empty_bar(s));
          else umma_commit<false>(empty_bar(s));
        }
        if (!ok) break;
        if (PAIR) umma_commit_pair(tfull_bar(acc));
        else umma_commit<false>(tfull_bar(acc));
      }
      if (!ok) {
        // Make sure no MMA is still writing TMEM before it is freed.
        umma_commit<PAIR>(drain_bar);
        volatile int no_abort = 0;
        mbar_wait_bounded(drain_bar, 0, kDrainLimitNs, p.err, ERRBIT_WAIT_DRAIN, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int ch = (warp - 2) >> 2;         // which half of the tile's columns
    constexpr int COLS = BN / (EPI_WARPS / 4);
    // Accumulator-free arrivals go to the even CTA, which issues the MMAs.
    const uint32_t te0 = PAIR ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    const uint32_t te1 = PAIR ? mapa_shared(tempty_bar(1), 0) : tempty_bar(1);
    const uint32_t stage = sStage + (uint32_t)(warp - 2) * 4096u;
    int lt = 0;
    for (int tile = first; tile < count; tile += stride, ++lt) {
      int g, m0, n0;
      coords(tile, rank, g, m0, n0);
      const int acc = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_ZSTATS) {
        // While the accumulator is still being computed: pull the tile's
        // bias columns into L1, so the epilogue's loads of them do not wait
        // on L2.  (Prefetching the residual rows measured slower.)
        const int n1 = n0 + ch * COLS;
        if (lane < (COLS * (int)sizeof(T)) / 128 && n1 + lane * (128 / (int)sizeof(T)) < p.N)
          prefetch_l1(reinterpret_cast<const T*>(p.bias) + (size_t)g * p.bias_gs + n1 + lane * (128 / sizeof(T)));
      }
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar(acc), aph, p.wait_limit_ns, p.err, ERRBIT_WAIT_EPILOGUE, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int m = m0 + q * 32 + lane;
      const int c0 = ch * COLS;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c0);
      ZSums zs[2] = {{0.f, 0.f, {0.f, 0.f}, {0.f, 0.f}}, {0.f, 0.f, {0.f, 0.f}, {0.f, 0.f}}};
      // The accumulator is released as soon as its last columns are in
      // registers, before they are converted and stored, so that the store
      // path never delays the next tile's MMAs.
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) mbar_arrive_remote(acc ? te1 : te0);
          else mbar_arrive(tempty_bar(acc));
        }
        released = true;
      };
      // A staged box is 32 rows x 128 bytes: 64 columns of a 16-bit output,
      // 32 of fp32 (two boxes per 64 columns).
      constexpr int OW = sizeof(T) == 4 ? 2 : 1;  // 32-bit words per output column pair
      for (int j0 = 0; j0 < COLS; j0 += 64) {
        if (n0 + c0 + j0 >= p.N || m0 + q * 32 >= p.M) break;  // warp-uniform
        uint32_t pk[32 * OW];
        {
          float v[64];
          tmem_ld_32x64(t_row + (uint32_t)j0, v);
          if (j0 + 64 >= COLS || n0 + c0 + j0 + 64 >= p.N) release();
          epilogue_convert<T, EPI>(p, g, m, n0 + c0 + j0, v, zs, pk);
          epilogue_convert<T, EPI>(p, g, m, n0 + c0 + j0 + 32, v + 32, zs, pk + 16 * OW);
        }
#pragma unroll
        for (int h = 0; h < OW; ++h) {
          const int nb = n0 + c0 + j0 + h * 32;
          if (h > 0 && nb >= p.N) break;  // warp-uniform
          // The previous box must have been read out of the staging buffer.
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          // Row `lane` of the box: eight 16-byte chunks, chunk j at position
          // j ^ (row % 8) (the tensor map's 128-byte swizzle).
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(stage + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), pk[32 * h + 4 * j],
                         pk[32 * h + 4 * j + 1], pk[32 * h + 4 * j + 2], pk[32 * h + 4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (KIND == GEMM_WGRAD) tma_store_3d(&tmC, stage, nb, m0 + q * 32, g);   // map {N, M, G}
            else tma_store_3d(&tmC, stage, nb, g, m0 + q * 32);                    // map {N, G, M}
            bulk_commit();
          }
        }
      }
      if (!released) release();
      if (EPI == EPI_BIAS_ZSTATS && m < p.M && n0 + c0 < p.N) {
        float4 w;
        const float s0 = zs[0].s.x + zs[0].s.y, q0 = zs[0].q.x + zs[0].q.y;
        const float s1 = zs[1].s.x + zs[1].s.y, q1 = zs[1].q.x + zs[1].q.y;
        w.x = zs[0].n > 0.f ? zs[0].k + s0 / zs[0].n : 0.f;
        w.y = zs[0].n > 0.f ? fmaxf(q0 - s0 * s0 / zs[0].n, 0.f) : 0.f;
        w.z = zs[1].n > 0.f ? zs[1].k + s1 / zs[1].n : 0.f;
        w.w = zs[1].n > 0.f ? fmaxf(q1 - s1 * s1 / zs[1].n, 0.f) : 0.f;
        const int grp = (n0 + c0) / kZStatsTile;
        *reinterpret_cast<float4*>(p.zstats + (((size_t)m * p.G + g) * p.zgroups + grp) * 4) = w;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // Pair: neither CTA leaves while the other may still read its shared
  // memory or signal its barriers, and TMEM is freed by both together.
  if (PAIR) cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

__global__ void k_bounded_wait_test(unsigned int* err, unsigned long long limit_ns) {
  pdl_enter();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must give up after limit_ns.
  if (threadIdx.x == 0)
    mbar_wait_bounded(smem_u32(&bar), 0, limit_ns, err, ERRBIT_WAIT_TEST, (volatile int*)&abort_flag);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Rank-3 tiled map with 128-byte swizzle; dims innermost first, strides in
// bytes for dims 1 and 2.
bool make_map(CUtensorMap* m, const void* base, int dtype, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
              uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapDataType dt = dtype == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Rank-5 map of an MN-major operand for the interleaved stage layout:
// element (mn, k, g) at mn * e + k * k_stride + g * g_stride bytes; dims
// {64, 8, MN / 64, K / 8, G}, box {64, 8, chunks, 8, 1} (one stage), 128-byte
// swizzle.  Needs MN % 64 == 0 and K % 8 == 0 (no box reaches past the
// tensor: K groups past K / 8 and chunks past MN / 64 are out of range and
// read as zero).
bool make_map_mn5(CUtensorMap* m, const void* base, int dtype, uint64_t mn, uint64_t k, uint64_t g,
                  uint64_t k_stride, uint64_t g_stride, uint32_t chunks) {
  auto enc = encode_fn();
  if (!enc || mn % 64 || k % 8) return false;
  cuuint64_t dims[5] = {64, 8, mn / 64, k / 8, g};
  cuuint64_t strides[4] = {k_stride, 128, 8 * k_stride, g_stride};
  cuuint32_t box[5] = {64, 8, chunks, BK / 8, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType dt = dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(m, dt, 5, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T, int KIND, int EPI, bool PAIR>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const Params& p,
                      cudaStream_t st) {
  auto k = k_gemm_tc<T, KIND, EPI, PAIR>;
  constexpr int SMEM_BYTES = Ring<PAIR>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (!PAIR) {
    const int grid = p.num_tiles < sm_count() ? p.num_tiles : sm_count();
    return launch_k(k, dim3(grid), dim3(THREADS), SMEM_BYTES, st, 1, a, b, c, p);
  }
  const int clusters = p.num_pair_tiles < sm_count() / 2 ? p.num_pair_tiles : sm_count() / 2;
  return launch_k(k, dim3(2 * (clusters > 0 ? clusters : 1)), dim3(THREADS), SMEM_BYTES, st, 2, a, b, c, p);
}

// fp32 operands (TF32 tensor cores): both operands K-major (the dgrad
// form); the caller stages transposed copies of MN-major operands.
template <bool PAIR>
cudaError_t dispatch_tf32(const GemmDesc& d, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                          const Params& p, cudaStream_t st) {
  switch (d.epi) {
    case EPI_STORE: return launch_tc<float, GEMM_DGRAD, EPI_STORE, PAIR>(a, b, c, p, st);
    case EPI_RESID: return launch_tc<float, GEMM_DGRAD, EPI_RESID, PAIR>(a, b, c, p, st);
    case EPI_BIAS_RESID: return launch_tc<float, GEMM_DGRAD, EPI_BIAS_RESID, PAIR>(a, b, c, p, st);
    case EPI_BIAS_ZSTATS: return launch_tc<float, GEMM_DGRAD, EPI_BIAS_ZSTATS, PAIR>(a, b, c, p, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, bool PAIR>
cudaError_t dispatch_tc(const GemmDesc& d, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const Params& p, cudaStream_t st) {
  switch (d.kind * 8 + d.epi) {
    case GEMM_FWD * 8 + EPI_STORE: return launch_tc<T, GEMM_FWD, EPI_STORE, PAIR>(a, b, c, p, st);
    case GEMM_FWD * 8 + EPI_BIAS: return launch_tc<T, GEMM_FWD, EPI_BIAS, PAIR>(a, b, c, p, st);
    case GEMM_FWD * 8 + EPI_BIAS_RESID: return launch_tc<T, GEMM_FWD, EPI_BIAS_RESID, PAIR>(a, b, c, p, st);
    case GEMM_FWD * 8 + EPI_BIAS_ZSTATS: return launch_tc<T, GEMM_FWD, EPI_BIAS_ZSTATS, PAIR>(a, b, c, p, st);
    case GEMM_DGRAD * 8 + EPI_STORE: return launch_tc<T, GEMM_DGRAD, EPI_STORE, PAIR>(a, b, c, p, st);
    case GEMM_DGRAD * 8 + EPI_RESID: return launch_tc<T, GEMM_DGRAD, EPI_RESID, PAIR>(a, b, c, p, st);
    case GEMM_WGRAD * 8 + EPI_STORE: return launch_tc<T, GEMM_WGRAD, EPI_STORE, PAIR>(a, b, c, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int sm_count() {
  static std::atomic<int> n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int c = n[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    c = v > 0 ? v : 1;
    n[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

bool gemm_tc_supported(const GemmDesc& d) {
  if (d.dtype != 0 && d.dtype != 1 && d.dtype != 2) return false;
  if (d.M <= 0 || d.N <= 0 || d.K <= 0 || d.G <= 0) return false;
  if (d.dtype == 0) {
    // TF32: K-major operands only (the dgrad form), 16-byte row strides.
    if (!d.tf32 || d.kind != GEMM_DGRAD || d.N % 8 || d.K % 4) return false;
    if ((d.a_rs | d.a_gs | d.c_rs | d.c_gs) % 4) return false;
    if (d.epi == EPI_BIAS_ZSTATS && (BN / (EPI_WARPS / 4) != kZStatsTile || !d.zstats || d.split % 8)) return false;
    return (d.epi == EPI_STORE || d.epi == EPI_RESID || d.epi == EPI_BIAS_RESID || d.epi == EPI_BIAS_ZSTATS) &&
           encode_fn() != nullptr;
  }
  if (d.a_rs || d.a_gs || d.c_rs || d.c_gs) return false;  // explicit strides: TF32 path only
  // 16-byte row strides for the tensor maps and the vector epilogue.  The
  // weight-gradient GEMMs reduce over K = B, the outermost dimension of both
  // operands' maps (no stride of its own); a ragged last k-block is
  // zero-filled by the copy.  K % 8 only selects the interleaved stages.
  if (d.N % 8 || (d.kind != GEMM_WGRAD && d.K % 8)) return false;
  if (d.kind == GEMM_WGRAD && d.M % 8) return false;
  if (d.epi == EPI_BIAS_ZSTATS && (BN / (EPI_WARPS / 4) != kZStatsTile || !d.zstats || d.split % 8)) return false;
  const int ok_epi = (d.kind == GEMM_FWD && (d.epi == EPI_STORE || d.epi == EPI_BIAS || d.epi == EPI_BIAS_RESID ||
                                             d.epi == EPI_BIAS_ZSTATS)) ||
                     (d.kind == GEMM_DGRAD && (d.epi == EPI_STORE || d.epi == EPI_RESID)) ||
                     (d.kind == GEMM_WGRAD && d.epi == EPI_STORE);
  return ok_epi && encode_fn() != nullptr;
}

cudaError_t gemm_tc_launch(const GemmDesc& d, unsigned int* err, cudaStream_t st) {
  if (!gemm_tc_supported(d)) return cudaErrorInvalidValue;
  const uint64_t e = d.dtype == 0 ? 4 : 2, M = d.M, N = d.N, K = d.K, G = d.G;
  const uint32_t BKE = (uint32_t)(128 / e);  // elements of a k-block
  // Paired mode whenever M spans at least two tiles (and the env switch
  // RMX_GEMM_PAIRS=0 is not set).
  static const bool pairs_on = [] {
    const char* v = getenv("RMX_GEMM_PAIRS");
    return !(v && v[0] == '0');
  }();
  const bool pair = pairs_on && d.M > BM;
  CUtensorMap ma, mb, mc;
  bool ok = true;
  const uint32_t b_chunks = (pair ? BN / 2 : BN) / 64;
  // Interleaved MN-major stages where the extents allow it (make_map_mn5
  // checks them; else the operand comes as separate 64-wide chunks through
  // rank-3 maps).
  bool il = true;
  // Activation rows [M, G, K] (defaults) or any (g, m) strides given.
  const uint64_t a_gs = d.a_gs ? (uint64_t)d.a_gs : K, a_rs = d.a_rs ? (uint64_t)d.a_rs : G * K;
  const uint64_t c_gs = d.c_gs ? (uint64_t)d.c_gs : N, c_rs = d.c_rs ? (uint64_t)d.c_rs : G * N;
  if (d.kind == GEMM_FWD || d.kind == GEMM_DGRAD) {
    ok &= make_map(&ma, d.A, d.dtype, K, G, M, a_gs * e, a_rs * e, BKE, 1, BM);       // A [M,G,K]
    if (d.kind == GEMM_FWD) {
      il = il && make_map_mn5(&mb, d.Bm, d.dtype, N, K, G, N * e, K * N * e, b_chunks);  // W [G,K,N]
      if (!il) ok &= make_map(&mb, d.Bm, d.dtype, N, K, G, N * e, K * N * e, 64, BK, 1);
    } else {
      ok &= make_map(&mb, d.Bm, d.dtype, K, N, G, K * e, N * K * e, BKE, pair ? BN / 2 : BN, 1);  // W [G,N,K]
    }
  } else {
    il = il && make_map_mn5(&ma, d.A, d.dtype, M, K, G, G * M * e, M * e, BM / 64) &&   // A [K,G,M]
         make_map_mn5(&mb, d.Bm, d.dtype, N, K, G, G * N * e, N * e, b_chunks);        // B [K,G,N]
    if (!il) {
      ok &= make_map(&ma, d.A, d.dtype, M, G, K, M * e, G * M * e, 64, 1, BK);
      ok &= make_map(&mb, d.Bm, d.dtype, N, G, K, N * e, G * N * e, 64, 1, BK);
    }
  }
  if (d.kind == GEMM_DGRAD) il = false;  // no MN-major operand
  // Output boxes of 32 rows x 64 columns, written by the epilogue warps.
  // (32 rows x 128 bytes: 64 columns of a 16-bit type, 32 of fp32.)
  if (d.kind == GEMM_WGRAD) ok &= make_map(&mc, d.C, d.dtype, N, M, G, N * e, M * N * e, BKE, 32, 1);  // C [G,M,N]
  else ok &= make_map(&mc, d.C, d.dtype, N, G, M, c_gs * e, c_rs * e, BKE, 1, 32);                    // C [M,G,N]
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.mn_il = il ? 1 : 0;
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.G = d.G;
  p.tiles_m = (d.M + BM - 1) / BM;
  p.tiles_n = (d.N + BN - 1) / BN;
  p.tiles_per_group = p.tiles_m * p.tiles_n;
  p.num_tiles = p.tiles_per_group * d.G;
  p.num_kb = (d.K + (int)BKE - 1) / (int)BKE;
  p.pairs_m = (p.tiles_m + 1) / 2;
  p.pair_tiles_per_group = p.pairs_m * p.tiles_n;
  p.num_pair_tiles = p.pair_tiles_per_group * d.G;
  p.out = d.C;
  if (d.kind == GEMM_WGRAD) {
    p.out_rs = d.N;
    p.out_gs = (long long)d.M * d.N;
  } else {
    p.out_rs = (long long)c_rs;
    p.out_gs = (long long)c_gs;
  }
  p.bias = d.bias;
  p.bias_gs = d.N;
  p.resid = d.resid;
  p.res_rs = p.out_rs;
  p.res_gs = p.out_gs;
  p.err = err;
  p.wait_limit_ns = kWaitLimitNs;
  p.zstats = d.zstats;
  p.split = d.split;
  p.zgroups = (d.N + kZStatsTile - 1) / kZStatsTile;
  if (d.dtype == 0) return pair ? dispatch_tf32<true>(d, ma, mb, mc, p, st) : dispatch_tf32<false>(d, ma, mb, mc, p, st);
  if (d.dtype == 1)
    return pair ? dispatch_tc<bf16, true>(d, ma, mb, mc, p, st) : dispatch_tc<bf16, false>(d, ma, mb, mc, p, st);
  return pair ? dispatch_tc<f16, true>(d, ma, mb, mc, p, st) : dispatch_tc<f16, false>(d, ma, mb, mc, p, st);
}

cudaError_t launch_bounded_wait_test(unsigned int* err, unsigned long long limit_ns, cudaStream_t st) {
  cudaError_t e = launch_k(k_bounded_wait_test, dim3(1), dim3(32), 0, st, 1, err, limit_ns);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool make_tensor_map_2d(CUtensorMap* m, const void* base, int dtype, uint64_t d0, uint64_t d1, uint64_t s1,
                        uint32_t b0, uint32_t b1) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {s1};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType dt = dtype == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace rmx
