// ls_grpo_loss_noalloc: the fused GRPO loss for callers that cannot allocate device memory.
//
// ls_grpo_loss needs a caller-provided device workspace of R doubles (the per-row loss
// terms that the fixed-order reduction sums).  Some callers cannot provide one: code that
// runs where cudaMalloc is off limits (inside a region that must not allocate because it
// is being captured or replayed as a fixed memory plan, an allocator that is not reentrant
// from the calling context, or a host process that may only hand over pointers to buffers
// it already owns).  This entry point takes the same inputs and outputs but keeps its
// scratch in a fixed array compiled into the library, so it calls no cudaMalloc, cudaFree
// or other allocating routine.
//
// The scratch array is a module global: every GPU that loads the library holds it
// (kNoAllocMaxRows doubles = 512 KB) until the process exits, and every call on a device
// shares it.  Calls whose kernels overlap on the GPU (different streams, or different host
// threads, without ordering between them) race on it; calls ordered on one stream do not.
// Every row term a call reads is written earlier by the same call (a row whose cluster
// exchange gave up a bounded wait writes NaN), so nothing needs to be cleared between calls.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/longstraw.h"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int64_t kNoAllocMaxRows = 65536;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) double g_noalloc_row_terms[kNoAllocMaxRows];

std::mutex g_mu;
double* g_scratch[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once per device
// with that device current.  In host code the array's name is only a host-side stand-in.
ls_status scratch_address(double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_last_error("cudaGetDevice failed in ls_grpo_loss_noalloc");
    return LS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_row_terms);
    if (e != cudaSuccess || p == nullptr) {
      set_last_error("cudaGetSymbolAddress of the no-allocation scratch failed");
      return LS_ERR_CUDA;
    }
    g_scratch[dev] = static_cast<double*>(p);
  }
  *out = g_scratch[dev];
  return LS_OK;
}

bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0u; }

}  // namespace
}  // namespace ls

extern "C" int64_t ls_grpo_loss_noalloc_max_rows(void) { return ls::kNoAllocMaxRows; }

extern "C" ls_status ls_grpo_loss_noalloc(int64_t R, int64_t V, int32_t G, const void* logits,
                                          const int32_t* ids, const float* logp_old,
                                          double advantage, double eps, double* loss_accum,
                                          void* dlogits, uint8_t* clip_mask, float* logp_out,
                                          void* stream) {
  using namespace ls;
  if (logits == nullptr || ids == nullptr || logp_old == nullptr || loss_accum == nullptr ||
      dlogits == nullptr || clip_mask == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  if (R < 1 || V < 1 || G < 1) return LS_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(advantage) || !(eps >= 0.0 && eps < 1.0))
    return LS_ERR_INVALID_ARGUMENT;
  if (R > kNoAllocMaxRows) {
    set_last_error("ls_grpo_loss_noalloc: R exceeds the fixed scratch capacity of 65536 rows");
    return LS_ERR_UNSUPPORTED;
  }
  if (V >= (int64_t(1) << 31)) return LS_ERR_UNSUPPORTED;
  if (!aligned_to(logits, 2) || !aligned_to(dlogits, 2) || !aligned_to(ids, 4) ||
      !aligned_to(logp_old, 4) || !aligned_to(loss_accum, 8) ||
      (logp_out != nullptr && !aligned_to(logp_out, 4)))
    return LS_ERR_MISALIGNED;
  // the same device and stream checks as ls_grpo_loss, before the scratch address of the
  // current device is looked up
  uint32_t* status = nullptr;
  ls_status st = static_cast<ls_status>(enter_call(stream, &status));
  if (st != LS_OK) return st;
  double* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != LS_OK) return st;
  LossArgs a{};
  a.R = R;
  a.V = V;
  a.G = G;
  a.logits = static_cast<const uint16_t*>(logits);
  a.ids = ids;
  a.logp_old = logp_old;
  a.A = advantage;
  a.eps = eps;
  a.loss_accum = loss_accum;
  a.dlogits = static_cast<uint16_t*>(dlogits);
  a.clip_mask = clip_mask;
  a.logp_out = logp_out;
  a.row_terms = scratch;
  a.status = status;
  cudaError_t e = injected_failure() ? cudaErrorLaunchFailure
                                     : launch_grpo_loss(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return static_cast<ls_status>(launch_failed(e, "grpo loss (no-allocation) launch"));
  return LS_OK;
}
