// No-allocation variant of the norm2 backward.
//
// Some callers cannot hand this library a scratch buffer: a host framework
// that owns every byte of device memory through its own pool and gives a
// plugin only its input and output tensors, or a deployment that must keep a
// fixed, known memory footprint and forbids allocations after start-up.  For
// them, rmx_ln2_backward_noalloc computes the norm2 backward (ds2 and the
// gamma2 / beta2 / bout gradients) with its partial-sum scratch in a
// fixed-size array that lives in this file as device global memory: it is
// reserved once per GPU when the library's module is loaded on that GPU and
// stays allocated until the process exits.  The entry point itself calls no
// cudaMalloc, cudaFree or other allocating routine.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call on each device looks up the
// real address with cudaGetSymbolAddress while that device is current, and
// every launch receives that pointer.

#include <atomic>

#include "../../include/rmx.h"
#include "common.cuh"
#include "kernels.h"

namespace rmx {
namespace {

// Capacity of the shared scratch array, in floats (16 MiB).
constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
// Cached device address per device.  Atomic because host threads may make
// their first call on the same device at the same time; they look up (and
// store) the same address, so whichever store lands is correct.
std::atomic<float*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once
// per device).  Returns nullptr if the lookup fails.
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  float* cached = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!cached) {
    float* p = nullptr;
    if (cudaGetSymbolAddress((void**)&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
    cached = p;
  }
  return cached;
}

bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace rmx

using namespace rmx;

extern "C" rmx_status rmx_ln2_backward_noalloc(const rmx_config* cfg, const void* dy, const void* s2,
                                               const float* mean2, const float* rstd2, const void* gamma2,
                                               void* ds2, void* dgamma2, void* dbeta2, void* dbout,
                                               rmx_stream stream) {
  if (!cfg || cfg->B < 1 || cfg->T < 1 || cfg->D < 1 || cfg->H < 1 || cfg->D % cfg->T) return RMX_ERR_INVALID_ARG;
  if (cfg->dtype != RMX_F32 && cfg->dtype != RMX_BF16 && cfg->dtype != RMX_F16) return RMX_ERR_INVALID_ARG;
  const void* ptrs[] = {dy, s2, mean2, rstd2, gamma2, ds2, dgamma2, dbeta2, dbout};
  for (const void* p : ptrs) {
    if (!p) return RMX_ERR_INVALID_ARG;
    if (!ok16(p)) return RMX_ERR_ALIGNMENT;
  }
  const int e = cfg->dtype == RMX_F32 ? 4 : 2;
  const int V = 16 / e;
  if (cfg->D % V || cfg->D / V > kRowThreadsMax) return RMX_ERR_UNSUPPORTED;

  // Partial sums per block of up to 64 samples: gamma2 and beta2
  // [nbblk*T, D] and bout [nbblk, T*D].  Shapes whose partial sums exceed the
  // array are rejected.
  RowArgs ra;
  ra.B = cfg->B;
  ra.T = cfg->T;
  ra.D = cfg->D;
  ra.H = cfg->H;
  ra.Dl = cfg->D;
  ra.Hl = cfg->H;
  ra.dtype = cfg->dtype;
  ra.nb_ln = cfg->B < 64 ? cfg->B : 64;
  ra.nbblk_ln = (cfg->B + ra.nb_ln - 1) / ra.nb_ln;
  ra.nb = ra.nb_ln;
  ra.nbblk = ra.nbblk_ln;
  if ((size_t)3 * ra.nbblk_ln * cfg->T * cfg->D > kNoAllocScratchFloats) return RMX_ERR_UNSUPPORTED;

  float* scratch = scratch_on_current_device();
  if (!scratch) return RMX_ERR_CUDA;
  const size_t P = (size_t)ra.nbblk_ln * cfg->T;
  float* pg2 = scratch;
  float* pb2 = pg2 + P * cfg->D;
  float* pbo = pb2 + P * cfg->D;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Every partial the column sums read is written by launch_ln2_bwd in this
  // same call, so nothing in the array has to start at zero.
  if (launch_ln2_bwd(ra, dy, s2, mean2, rstd2, gamma2, ds2, pg2, pb2, pbo, st) != cudaSuccess) return RMX_ERR_CUDA;
  ColsumJob jobs[3] = {
      {pg2, dgamma2, (int)P, cfg->D},
      {pb2, dbeta2, (int)P, cfg->D},
      {pbo, dbout, ra.nbblk_ln, cfg->T * cfg->D},
  };
  if (launch_colsums(jobs, 3, cfg->dtype, st) != cudaSuccess) return RMX_ERR_CUDA;
  return RMX_OK;
}
