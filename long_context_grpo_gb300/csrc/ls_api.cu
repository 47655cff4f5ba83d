// Host side of the C ABI declared in include/longstraw.h: argument validation, TMA
// descriptor encoding, launch sequencing on the caller's stream and error mapping.
// The library allocates no device memory; the only device-resident state it owns is the
// 4-byte status word below (one per device, a module global).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/longstraw.h"
#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {

__device__ uint32_t g_status_word = 0u;

// ----- launch-failure injection (ls_debug_fail_launch): a countdown of launch attempts;
// the attempt that finds it at 0 is not made and reports LS_ERR_CUDA.
std::atomic<int64_t> g_fail_countdown{-1};
thread_local bool t_injected = false;

bool injected_failure() {
  int64_t c = g_fail_countdown.load();
  while (c >= 0) {
    if (g_fail_countdown.compare_exchange_weak(c, c - 1)) {
      if (c != 0) return false;
      t_injected = true;
      return true;
    }
  }
  return false;
}

namespace {

constexpr uint32_t kMagic = 0x4c535046u;  // "LSPF"
constexpr int kMaxDevices = 64;

thread_local char t_last_error[256] = "";

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

std::mutex g_dev_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

ls_status cuda_fail(cudaError_t e, const char* what) {
  if (t_injected) {
    t_injected = false;
    snprintf(t_last_error, sizeof(t_last_error), "%s: launch failure injected by ls_debug_fail_launch",
             what);
    return LS_ERR_CUDA;
  }
  snprintf(t_last_error, sizeof(t_last_error), "%s: %s", what, cudaGetErrorString(e));
  return LS_ERR_CUDA;
}

// One NVTX range per API call (visible to profilers; no-op without one attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }
bool aligned_n(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0u; }

ls_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return LS_ERR_UNSUPPORTED;
  return LS_OK;
}

// Address of this device's status word (looked up once per device, with it current).
ls_status status_ptr(int dev, uint32_t** out) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_status_ptr[dev];
  return LS_OK;
}

ls_status check_stream(void* stream, int dev) {
  if (stream == nullptr) return LS_OK;
  int sdev = -1;
  cudaError_t e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetDevice");
  return sdev == dev ? LS_OK : LS_ERR_WRONG_DEVICE;
}

ls_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) {
    snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled unavailable");
    return LS_ERR_CUDA;
  }
  return LS_OK;
}

// 3-D bf16 THD tensor [T][H][D] with a {64, hbox, tbox} box and 128-byte swizzle.
ls_status encode_thd(CUtensorMap* m, const void* base, int64_t T, int H, int D, int hbox,
                     int tbox) {
  ls_status st = get_encoder();
  if (st != LS_OK) return st;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(D) * 2u};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(hbox), static_cast<cuuint32_t>(tbox)};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (%d)",
             static_cast<int>(r));
    return LS_ERR_CUDA;
  }
  return LS_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----- optional per-launch timing (ls_timing_enable / ls_timing_read)
struct TimedLaunch {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mu;
bool g_timing = false;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_free_events;

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets the launches made during its lifetime when timing is enabled.
class LaunchTimer {
 public:
  LaunchTimer(int kernel, cudaStream_t s) : kernel_(kernel), s_(s) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (!g_timing) return;
    start_ = take_event();
    stop_ = take_event();
    if (start_ && stop_) cudaEventRecord(start_, s_);
  }
  ~LaunchTimer() {
    if (!start_ || !stop_) return;
    cudaEventRecord(stop_, s_);
    std::lock_guard<std::mutex> lk(g_timing_mu);
    g_timed.push_back({kernel_, start_, stop_});
  }

 private:
  int kernel_;
  cudaStream_t s_;
  cudaEvent_t start_ = nullptr, stop_ = nullptr;
};

}  // namespace

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

// Accessors for other translation units of the library (no change to any entry point).
void set_last_error(const char* msg) { snprintf(t_last_error, sizeof(t_last_error), "%s", msg); }

int launch_failed(cudaError_t e, const char* what) { return cuda_fail(e, what); }

}  // namespace ls

struct ls_prefix_s {
  uint32_t magic;
  int device;
  ls::AttnShape shape;    // R unused here
  const void* k_prefix;
  const void* v_prefix;
  float* dk_acc;
  float* dv_acc;
  CUtensorMap tm_k;     // box {64, 1, 128}: every 128-key tile of the prompt
  CUtensorMap tm_v;
};

namespace {

using namespace ls;

ls_status check_handle(ls_prefix_t h) {
  if (h == nullptr || h->magic != kMagic) return LS_ERR_NOT_PREPARED;
  return LS_OK;
}

ls_status enter(ls_prefix_t h, void* stream, uint32_t** status) {
  int dev = 0;
  ls_status st = current_device(&dev);
  if (st != LS_OK) return st;
  if (h != nullptr && dev != h->device) return LS_ERR_WRONG_DEVICE;
  st = check_stream(stream, dev);
  if (st != LS_OK) return st;
  return status_ptr(dev, status);
}

}  // namespace

namespace ls {
int enter_call(void* stream, uint32_t** status) { return enter(nullptr, stream, status); }
}  // namespace ls

namespace {

// Rows [row0, ...) of a prefix-shaped bf16 [P, Hkv, D] buffer.
const void* block_rows(ls_prefix_t h, const void* base, int64_t row0) {
  return static_cast<const uint16_t*>(base) + row0 * h->shape.Hkv * h->shape.D;
}

// Packed-response offsets: 1 <= G <= kMaxPacked, cu[0] = 0, strictly increasing, total
// below 2^31.
ls_status check_cu(int32_t G, const int64_t* cu) {
  if (cu == nullptr || G < 1) return LS_ERR_INVALID_ARGUMENT;
  if (G > kMaxPacked) return LS_ERR_UNSUPPORTED;
  if (cu[0] != 0) return LS_ERR_INVALID_ARGUMENT;
  for (int b = 0; b < G; ++b)
    if (cu[b + 1] <= cu[b]) return LS_ERR_INVALID_ARGUMENT;
  if (cu[G] >= (int64_t(1) << 31)) return LS_ERR_UNSUPPORTED;
  return LS_OK;
}

size_t bwd_workspace_bytes(ls_prefix_t h, int32_t G, const int64_t* cu) {
  int64_t n_qt = 0;
  for (int b = 0; b < G; ++b) n_qt += (cu[b + 1] - cu[b] + h->shape.qt - 1) / h->shape.qt;
  return align_up(static_cast<size_t>(h->shape.Hkv) * n_qt * 256 * sizeof(float), 256);
}

// Replay forward of the packed responses cu (G of them, total rows cu[G]) against the first
// P_eff rows of the handle's prefix.
ls_status replay_fwd_impl(ls_prefix_t h, int64_t P_eff, int32_t G, const int64_t* cu,
                          const void* q, const void* k_suffix, const void* v_suffix, void* o,
                          float* lse, void* stream, int no_suffix = 0) {
  if (q == nullptr || k_suffix == nullptr || v_suffix == nullptr || o == nullptr ||
      lse == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  ls_status st = check_cu(G, cu);
  if (st != LS_OK) return st;
  const int64_t R = cu[G];
  if (!aligned16(q) || !aligned16(k_suffix) || !aligned16(v_suffix) || !aligned16(o) ||
      !aligned_n(lse, 4))
    return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  st = enter(h, stream, &status);
  if (st != LS_OK) return st;

  FwdArgs a{};
  a.sh = h->shape;
  a.sh.P = P_eff;
  a.sh.R = R;
  varlen_build(&a.vl, G, cu, a.sh.qt);
  a.tm_kp = &h->tm_k;
  a.tm_vp = &h->tm_v;
  const AttnShape& sh = a.sh;
  st = encode_thd(&a.tm_q, q, R, sh.Hq, sh.D, sh.g, sh.qt);
  if (no_suffix) {
    a.tm_ks = h->tm_k;   // never read: prompt keys only
    a.tm_vs = h->tm_v;
  } else {
    if (st == LS_OK) st = encode_thd(&a.tm_ks, k_suffix, R, sh.Hkv, sh.D, 1, 128);
    if (st == LS_OK) st = encode_thd(&a.tm_vs, v_suffix, R, sh.Hkv, sh.D, 1, 128);
  }
  if (st != LS_OK) return st;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.no_suffix = no_suffix;
  a.status = status;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_REPLAY_FWD, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_attn_fwd(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "replay forward launch");
}

// Replay backward of the packed responses against the first P_eff prefix rows.
// suffix_to_acc (one response only): the suffix keys' gradients go into the accumulators at
// rows P_eff + key (dk/dv_suffix unused).
ls_status replay_bwd_impl(ls_prefix_t h, int64_t P_eff, int32_t G, const int64_t* cu,
                          const void* q, const void* k_suffix, const void* v_suffix,
                          const void* o, const float* lse, const void* d_out, void* dq,
                          void* dk_suffix, void* dv_suffix, int suffix_to_acc, void* workspace,
                          size_t workspace_bytes, void* stream, int no_suffix = 0) {
  if (q == nullptr || k_suffix == nullptr || v_suffix == nullptr || o == nullptr ||
      lse == nullptr || d_out == nullptr || dq == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  ls_status st = check_cu(G, cu);
  if (st != LS_OK) return st;
  if (suffix_to_acc && G != 1) return LS_ERR_INVALID_ARGUMENT;
  const int64_t R = cu[G];
  if (workspace == nullptr || workspace_bytes < bwd_workspace_bytes(h, G, cu))
    return LS_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_suffix) || !aligned16(v_suffix) || !aligned16(o) ||
      !aligned16(d_out) || !aligned16(dq) || !aligned16(workspace) || !aligned_n(lse, 4))
    return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  st = enter(h, stream, &status);
  if (st != LS_OK) return st;

  BwdArgs a{};
  a.sh = h->shape;
  a.sh.P = P_eff;
  a.sh.R = R;
  varlen_build(&a.vl, G, cu, a.sh.qt);
  a.tm_kp = &h->tm_k;
  a.tm_vp = &h->tm_v;
  const AttnShape& sh = a.sh;
  st = encode_thd(&a.tm_q, q, R, sh.Hq, sh.D, sh.g, sh.qt);
  if (st == LS_OK) st = encode_thd(&a.tm_do, d_out, R, sh.Hq, sh.D, sh.g, sh.qt);
  if (no_suffix) {
    a.tm_ks = h->tm_k;   // never read: prompt keys only
    a.tm_vs = h->tm_v;
  } else {
    if (st == LS_OK) st = encode_thd(&a.tm_ks, k_suffix, R, sh.Hkv, sh.D, 1, 128);
    if (st == LS_OK) st = encode_thd(&a.tm_vs, v_suffix, R, sh.Hkv, sh.D, 1, 128);
  }
  if (st != LS_OK) return st;
  float* rowstats = static_cast<float*>(workspace);
  a.rowstats = rowstats;
  a.dq = static_cast<uint16_t*>(dq);
  a.dk_suf = static_cast<uint16_t*>(dk_suffix);
  a.dv_suf = static_cast<uint16_t*>(dv_suffix);
  a.dk_acc = h->dk_acc;
  a.dv_acc = h->dv_acc;
  a.suffix_to_acc = suffix_to_acc;
  a.no_suffix = no_suffix;
  a.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_BWD_PREP, s);
    e = injected_failure() ? cudaErrorLaunchFailure : launch_bwd_prep(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(d_out), lse,
                        rowstats, sh, a.vl, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "replay backward prep launch");
  {
    LaunchTimer t(LS_KERNEL_BWD_DKDV, s);
    e = injected_failure() ? cudaErrorLaunchFailure : launch_attn_bwd_dkdv(a, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "replay backward dK/dV launch");
  {
    LaunchTimer t(LS_KERNEL_BWD_DQ, s);
    e = injected_failure() ? cudaErrorLaunchFailure : launch_attn_bwd_dq(a, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "replay backward dQ launch");
  return LS_OK;
}

// out = scale * acc over accumulator rows [row0, row0 + nrows) (fp32 or bf16 out, optional
// reset), or acc *= scale in place when both outputs are NULL.
ls_status finalize_impl(ls_prefix_t h, int64_t row0, int64_t nrows, float scale, void* dk_out,
                        void* dv_out, int out_is_fp32, int reset_acc, void* stream) {
  if (!std::isfinite(scale)) return LS_ERR_INVALID_ARGUMENT;
  if ((dk_out == nullptr) != (dv_out == nullptr)) return LS_ERR_INVALID_ARGUMENT;
  const bool inplace = dk_out == nullptr;
  if (inplace && reset_acc) return LS_ERR_INVALID_ARGUMENT;
  if (!inplace && (!aligned16(dk_out) || !aligned16(dv_out))) return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  ls_status st = enter(h, stream, &status);
  if (st != LS_OK) return st;
  const size_t row = static_cast<size_t>(h->shape.Hkv) * h->shape.D;
  const size_t n = static_cast<size_t>(nrows) * row;
  float* dk = h->dk_acc + static_cast<size_t>(row0) * row;
  float* dv = h->dv_acc + static_cast<size_t>(row0) * row;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  LaunchTimer t(LS_KERNEL_FINALIZE, s);
  if (inplace) {
    e = injected_failure() ? cudaErrorLaunchFailure : launch_scale_inplace(dk, n, scale, s);
    if (e == cudaSuccess) e = injected_failure() ? cudaErrorLaunchFailure : launch_scale_inplace(dv, n, scale, s);
  } else {
    e = injected_failure() ? cudaErrorLaunchFailure : launch_finalize(dk, dk_out, n, scale, out_is_fp32 ? 1 : 0, reset_acc ? 1 : 0, s);
    if (e == cudaSuccess)
      e = injected_failure() ? cudaErrorLaunchFailure : launch_finalize(dv, dv_out, n, scale, out_is_fp32 ? 1 : 0, reset_acc ? 1 : 0, s);
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "finalize launch");
}

}  // namespace

extern "C" {

const char* ls_version(void) { return "0.1.0"; }

const char* ls_last_error(void) { return t_last_error; }

const char* ls_status_string(ls_status s) {
  switch (s) {
    case LS_OK: return "ok";
    case LS_ERR_INVALID_ARGUMENT: return "invalid argument";
    case LS_ERR_UNSUPPORTED: return "unsupported shape";
    case LS_ERR_NOT_PREPARED: return "prefix handle not prepared";
    case LS_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case LS_ERR_CUDA: return "CUDA error";
    case LS_ERR_TIMEOUT: return "device wait timed out";
    case LS_ERR_DEVICE_STATUS: return "device-side check failed";
    case LS_ERR_WORKSPACE: return "workspace missing or too small";
    case LS_ERR_WRONG_DEVICE: return "wrong device";
  }
  return "unknown status";
}

ls_status ls_prefix_prepare(const ls_prefix_desc* d, ls_prefix_t* out, void* stream) {
  NvtxRange nvtx_range("ls_prefix_prepare");
  if (d == nullptr || out == nullptr) return LS_ERR_INVALID_ARGUMENT;
  if (d->k_prefix == nullptr || d->v_prefix == nullptr || d->dk_acc == nullptr ||
      d->dv_acc == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  if (d->P < 1 || d->Hq < 1 || d->Hkv < 1) return LS_ERR_INVALID_ARGUMENT;
  if (!(d->softmax_scale >= 0.0f) || !std::isfinite(d->softmax_scale))
    return LS_ERR_INVALID_ARGUMENT;
  if (d->D != 64 && d->D != 128) return LS_ERR_UNSUPPORTED;
  if (d->Hq % d->Hkv != 0) return LS_ERR_UNSUPPORTED;
  const int g = d->Hq / d->Hkv;
  if (g > 16) return LS_ERR_UNSUPPORTED;
  if (d->P >= (int64_t(1) << 31)) return LS_ERR_UNSUPPORTED;
  if (!aligned16(d->k_prefix) || !aligned16(d->v_prefix) || !aligned16(d->dk_acc) ||
      !aligned16(d->dv_acc))
    return LS_ERR_MISALIGNED;

  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  int dev = 0;
  cudaGetDevice(&dev);

  ls_prefix_s* h = new (std::nothrow) ls_prefix_s();
  if (h == nullptr) return LS_ERR_INVALID_ARGUMENT;
  h->device = dev;
  h->shape.P = d->P;
  h->shape.R = 0;
  h->shape.Hq = d->Hq;
  h->shape.Hkv = d->Hkv;
  h->shape.D = d->D;
  h->shape.g = g;
  h->shape.qt = 128 / g;
  h->shape.scale = d->softmax_scale > 0.0f ? d->softmax_scale
                                           : 1.0f / std::sqrt(static_cast<float>(d->D));
  h->k_prefix = d->k_prefix;
  h->v_prefix = d->v_prefix;
  h->dk_acc = d->dk_acc;
  h->dv_acc = d->dv_acc;
  st = encode_thd(&h->tm_k, d->k_prefix, d->P, d->Hkv, d->D, 1, 128);
  if (st == LS_OK) st = encode_thd(&h->tm_v, d->v_prefix, d->P, d->Hkv, d->D, 1, 128);
  if (st != LS_OK) {
    delete h;
    return st;
  }
  const size_t n = static_cast<size_t>(d->P) * d->Hkv * d->D;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_ZERO, s);
    e = injected_failure() ? cudaErrorLaunchFailure : launch_zero_f32(d->dk_acc, n, s);
    if (e == cudaSuccess) e = injected_failure() ? cudaErrorLaunchFailure : launch_zero_f32(d->dv_acc, n, s);
  }
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "prefix accumulator zeroing");
  }
  h->magic = kMagic;
  *out = h;
  return LS_OK;
}

ls_status ls_prefix_destroy(ls_prefix_t h) {
  if (h == nullptr) return LS_OK;
  if (h->magic != kMagic) return LS_ERR_NOT_PREPARED;
  h->magic = 0;
  delete h;
  return LS_OK;
}

ls_status ls_replay_fwd(ls_prefix_t h, int64_t R, const void* q, const void* k_suffix,
                        const void* v_suffix, void* o, float* lse, void* stream) {
  NvtxRange nvtx_range("ls_replay_fwd");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  const int64_t cu[2] = {0, R};
  if (R < 1) return LS_ERR_INVALID_ARGUMENT;
  return replay_fwd_impl(h, h->shape.P, 1, cu, q, k_suffix, v_suffix, o, lse, stream);
}

ls_status ls_replay_fwd_packed(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens,
                               const void* q, const void* k_suffix, const void* v_suffix,
                               void* o, float* lse, void* stream) {
  NvtxRange nvtx_range("ls_replay_fwd_packed");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  return replay_fwd_impl(h, h->shape.P, G, cu_seqlens, q, k_suffix, v_suffix, o, lse, stream);
}

ls_status ls_block_replay_fwd(ls_prefix_t h, int64_t prefix_len, int64_t R, const void* q,
                              void* o, float* lse, void* stream) {
  NvtxRange nvtx_range("ls_block_replay_fwd");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (prefix_len < 1 || R < 1 || prefix_len > h->shape.P - R) return LS_ERR_INVALID_ARGUMENT;
  const int64_t cu[2] = {0, R};
  return replay_fwd_impl(h, prefix_len, 1, cu, q, block_rows(h, h->k_prefix, prefix_len),
                         block_rows(h, h->v_prefix, prefix_len), o, lse, stream);
}

size_t ls_replay_bwd_workspace_bytes(ls_prefix_t h, int64_t R) {
  if (check_handle(h) != LS_OK || R < 1) return 0;
  const int64_t cu[2] = {0, R};
  return bwd_workspace_bytes(h, 1, cu);
}

ls_status ls_replay_bwd(ls_prefix_t h, int64_t R, const void* q, const void* k_suffix,
                        const void* v_suffix, const void* o, const float* lse,
                        const void* d_out, void* dq, void* dk_suffix, void* dv_suffix,
                        void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("ls_replay_bwd");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (dk_suffix == nullptr || dv_suffix == nullptr) return LS_ERR_INVALID_ARGUMENT;
  if (!aligned16(dk_suffix) || !aligned16(dv_suffix)) return LS_ERR_MISALIGNED;
  if (R < 1) return LS_ERR_INVALID_ARGUMENT;
  const int64_t cu[2] = {0, R};
  return replay_bwd_impl(h, h->shape.P, 1, cu, q, k_suffix, v_suffix, o, lse, d_out, dq,
                         dk_suffix, dv_suffix, 0, workspace, workspace_bytes, stream);
}

size_t ls_replay_bwd_packed_workspace_bytes(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens) {
  if (check_handle(h) != LS_OK || check_cu(G, cu_seqlens) != LS_OK) return 0;
  return bwd_workspace_bytes(h, G, cu_seqlens);
}

ls_status ls_replay_bwd_packed(ls_prefix_t h, int32_t G, const int64_t* cu_seqlens,
                               const void* q, const void* k_suffix, const void* v_suffix,
                               const void* o, const float* lse, const void* d_out, void* dq,
                               void* dk_suffix, void* dv_suffix, void* workspace,
                               size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("ls_replay_bwd_packed");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (dk_suffix == nullptr || dv_suffix == nullptr) return LS_ERR_INVALID_ARGUMENT;
  if (!aligned16(dk_suffix) || !aligned16(dv_suffix)) return LS_ERR_MISALIGNED;
  return replay_bwd_impl(h, h->shape.P, G, cu_seqlens, q, k_suffix, v_suffix, o, lse, d_out,
                         dq, dk_suffix, dv_suffix, 0, workspace, workspace_bytes, stream);
}

ls_status ls_block_replay_bwd(ls_prefix_t h, int64_t prefix_len, int64_t R, const void* q,
                              const void* o, const float* lse, const void* d_out, void* dq,
                              void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("ls_block_replay_bwd");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (prefix_len < 1 || R < 1 || prefix_len > h->shape.P - R) return LS_ERR_INVALID_ARGUMENT;
  const int64_t cu[2] = {0, R};
  return replay_bwd_impl(h, prefix_len, 1, cu, q, block_rows(h, h->k_prefix, prefix_len),
                         block_rows(h, h->v_prefix, prefix_len), o, lse, d_out, dq, nullptr,
                         nullptr, 1, workspace, workspace_bytes, stream);
}

size_t ls_grpo_loss_workspace_bytes(int64_t R) {
  if (R < 1) return 0;
  return align_up(static_cast<size_t>(R) * sizeof(double), 256);
}

ls_status ls_grpo_loss(int64_t R, int64_t V, int32_t G, const void* logits, const int32_t* ids,
                       const float* logp_old, double advantage, double eps, double* loss_accum,
                       void* dlogits, uint8_t* clip_mask, float* logp_out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("ls_grpo_loss");
  if (logits == nullptr || ids == nullptr || logp_old == nullptr || loss_accum == nullptr ||
      dlogits == nullptr || clip_mask == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  if (R < 1 || V < 1 || G < 1) return LS_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(advantage) || !(eps >= 0.0 && eps < 1.0)) return LS_ERR_INVALID_ARGUMENT;
  if (R >= (int64_t(1) << 31) || V >= (int64_t(1) << 31)) return LS_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < ls_grpo_loss_workspace_bytes(R))
    return LS_ERR_WORKSPACE;
  if (!aligned_n(logits, 2) || !aligned_n(dlogits, 2) || !aligned_n(ids, 4) ||
      !aligned_n(logp_old, 4) || !aligned_n(loss_accum, 8) || !aligned16(workspace) ||
      (logp_out != nullptr && !aligned_n(logp_out, 4)))
    return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
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
  a.row_terms = static_cast<double*>(workspace);
  a.status = status;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_GRPO_LOSS, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_grpo_loss(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "grpo loss launch");
}

ls_status ls_token_logp(int64_t R, int64_t V, const void* logits, const int32_t* ids,
                        float* logp_out, void* stream) {
  NvtxRange nvtx_range("ls_token_logp");
  if (logits == nullptr || ids == nullptr || logp_out == nullptr) return LS_ERR_INVALID_ARGUMENT;
  if (R < 1 || V < 1) return LS_ERR_INVALID_ARGUMENT;
  if (R >= (int64_t(1) << 31) || V >= (int64_t(1) << 31)) return LS_ERR_UNSUPPORTED;
  if (!aligned_n(logits, 2) || !aligned_n(ids, 4) || !aligned_n(logp_out, 4))
    return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  LossArgs a{};
  a.R = R;
  a.V = V;
  a.G = 1;
  a.logits = static_cast<const uint16_t*>(logits);
  a.ids = ids;
  a.logp_out = logp_out;
  a.status = status;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_TOKEN_LOGP, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_token_logp(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "token log-prob launch");
}

ls_status ls_replay_fwd_prompt_only(ls_prefix_t h, int64_t R, const void* q, void* o, float* lse,
                                    void* stream) {
  NvtxRange nvtx_range("ls_replay_fwd_prompt_only");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (R < 1) return LS_ERR_INVALID_ARGUMENT;
  const int64_t cu[2] = {0, R};
  return replay_fwd_impl(h, h->shape.P, 1, cu, q, h->k_prefix, h->v_prefix, o, lse, stream, 1);
}

ls_status ls_replay_bwd_prompt_only(ls_prefix_t h, int64_t R, const void* q, const void* o,
                                    const float* lse, const void* d_out, void* dq,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("ls_replay_bwd_prompt_only");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (R < 1) return LS_ERR_INVALID_ARGUMENT;
  const int64_t cu[2] = {0, R};
  return replay_bwd_impl(h, h->shape.P, 1, cu, q, h->k_prefix, h->v_prefix, o, lse, d_out, dq,
                         nullptr, nullptr, 0, workspace, workspace_bytes, stream, 1);
}

ls_status ls_attn_merge(int32_t n, int64_t R, int32_t Hq, int32_t D, const void* const* o_parts,
                        const float* const* lse_parts, void* o, float* lse, void* stream) {
  NvtxRange nvtx_range("ls_attn_merge");
  if (o_parts == nullptr || lse_parts == nullptr || o == nullptr || lse == nullptr)
    return LS_ERR_INVALID_ARGUMENT;
  if (n < 1 || R < 1 || Hq < 1 || D < 8) return LS_ERR_INVALID_ARGUMENT;
  if (n > kMaxParts || D % 8 != 0) return LS_ERR_UNSUPPORTED;
  MergeArgs a{};
  a.n = n;
  a.rows = R * Hq;
  a.D = D;
  for (int r = 0; r < n; ++r) {
    if (o_parts[r] == nullptr || lse_parts[r] == nullptr) return LS_ERR_INVALID_ARGUMENT;
    if (!aligned16(o_parts[r]) || !aligned_n(lse_parts[r], 4)) return LS_ERR_MISALIGNED;
    a.o_parts[r] = static_cast<const uint16_t*>(o_parts[r]);
    a.lse_parts[r] = lse_parts[r];
  }
  if (!aligned16(o) || !aligned_n(lse, 4)) return LS_ERR_MISALIGNED;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_MERGE, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_attn_merge(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "merge launch");
}

ls_status ls_sum_bf16(int32_t n, int64_t count, const void* const* parts, void* out, void* stream) {
  NvtxRange nvtx_range("ls_sum_bf16");
  if (parts == nullptr || out == nullptr || n < 1 || count < 1) return LS_ERR_INVALID_ARGUMENT;
  if (n > kMaxParts || count % 8 != 0) return LS_ERR_UNSUPPORTED;
  SumArgs a{};
  a.n = n;
  a.count = count;
  for (int r = 0; r < n; ++r) {
    if (parts[r] == nullptr) return LS_ERR_INVALID_ARGUMENT;
    if (!aligned16(parts[r])) return LS_ERR_MISALIGNED;
    a.parts[r] = static_cast<const uint16_t*>(parts[r]);
  }
  if (!aligned16(out)) return LS_ERR_MISALIGNED;
  a.out = static_cast<uint16_t*>(out);
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_SUM, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_sum_bf16(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "sum launch");
}

ls_status ls_bf16_to_f32(int64_t count, const void* in, float* out, void* stream) {
  NvtxRange nvtx_range("ls_bf16_to_f32");
  if (in == nullptr || out == nullptr || count < 1) return LS_ERR_INVALID_ARGUMENT;
  if (count % 8 != 0) return LS_ERR_UNSUPPORTED;
  if (!aligned16(in) || !aligned16(out)) return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_CAST, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_bf16_to_f32(in, out, static_cast<size_t>(count), static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "bf16 -> fp32 launch");
}

ls_status ls_f32_to_bf16(int64_t count, const float* in, void* out, void* stream) {
  NvtxRange nvtx_range("ls_f32_to_bf16");
  if (in == nullptr || out == nullptr || count < 1) return LS_ERR_INVALID_ARGUMENT;
  if (count % 8 != 0) return LS_ERR_UNSUPPORTED;
  if (!aligned16(in) || !aligned16(out)) return LS_ERR_MISALIGNED;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  cudaError_t e;
  {
    LaunchTimer t(LS_KERNEL_CAST, static_cast<cudaStream_t>(stream));
    e = injected_failure() ? cudaErrorLaunchFailure : launch_f32_to_bf16(in, out, static_cast<size_t>(count), static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "fp32 -> bf16 launch");
}

ls_status ls_prefix_grad_finalize(ls_prefix_t h, float scale, void* dk_out, void* dv_out,
                                  int out_is_fp32, int reset_acc, void* stream) {
  NvtxRange nvtx_range("ls_prefix_grad_finalize");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  return finalize_impl(h, 0, h->shape.P, scale, dk_out, dv_out, out_is_fp32, reset_acc, stream);
}

ls_status ls_prefix_grad_finalize_rows(ls_prefix_t h, int64_t row0, int64_t nrows, float scale,
                                       void* dk_out, void* dv_out, int out_is_fp32,
                                       int reset_acc, void* stream) {
  NvtxRange nvtx_range("ls_prefix_grad_finalize_rows");
  ls_status st = check_handle(h);
  if (st != LS_OK) return st;
  if (row0 < 0 || nrows < 1 || row0 > h->shape.P - nrows) return LS_ERR_INVALID_ARGUMENT;
  return finalize_impl(h, row0, nrows, scale, dk_out, dv_out, out_is_fp32, reset_acc, stream);
}

ls_status ls_debug_wait_timeout(uint64_t limit_ns, void* stream) {
  NvtxRange nvtx_range("ls_debug_wait_timeout");
  if (limit_ns == 0 || limit_ns > 10000000000ull) return LS_ERR_INVALID_ARGUMENT;
  uint32_t* status = nullptr;
  ls_status st = enter(nullptr, stream, &status);
  if (st != LS_OK) return st;
  cudaError_t e = injected_failure() ? cudaErrorLaunchFailure : launch_wait_timeout(limit_ns, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LS_OK : cuda_fail(e, "wait-timeout self test launch");
}

ls_status ls_debug_fail_launch(int64_t after) {
  g_fail_countdown.store(after < 0 ? -1 : after);
  return LS_OK;
}

int64_t ls_debug_fail_launch_pending(void) { return g_fail_countdown.load(); }

ls_status ls_timing_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing = enable != 0;
  return LS_OK;
}

ls_status ls_timing_read(double* total_ms, int64_t* launches, int n) {
  if (total_ms == nullptr || launches == nullptr || n < LS_KERNEL_COUNT)
    return LS_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n; ++i) {
    total_ms[i] = 0.0;
    launches[i] = 0;
  }
  std::vector<TimedLaunch> done;
  {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    done.swap(g_timed);
  }
  ls_status st = LS_OK;
  for (const TimedLaunch& t : done) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "timing event");
    } else {
      total_ms[t.kernel] += ms;
      launches[t.kernel] += 1;
    }
  }
  std::lock_guard<std::mutex> lk(g_timing_mu);
  for (const TimedLaunch& t : done) {
    g_free_events.push_back(t.start);
    g_free_events.push_back(t.stop);
  }
  return st;
}

ls_status ls_get_device_status(void* stream, uint32_t* bits) {
  NvtxRange nvtx_range("ls_get_device_status");
  int dev = 0;
  ls_status st = current_device(&dev);
  if (st != LS_OK) return st;
  uint32_t* sp = nullptr;
  st = status_ptr(dev, &sp);
  if (st != LS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0, zero = 0;
  cudaError_t e = cudaMemcpyAsync(&host, sp, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sp, &zero, sizeof(zero), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  if (bits != nullptr) *bits = host;
  if (host & DEV_WAIT_TIMEOUT) return LS_ERR_TIMEOUT;
  if (host != 0u) return LS_ERR_DEVICE_STATUS;
  return LS_OK;
}

}  // extern "C"
