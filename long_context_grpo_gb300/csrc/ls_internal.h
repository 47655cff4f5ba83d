// Internal launch interface between the C-ABI host layer (ls_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ls {

// ----- GRPO loss (k_loss.cu)
struct LossArgs {
  int64_t R, V;
  int32_t G;
  const uint16_t* logits;   // bf16 [R, V]
  const int32_t* ids;       // [R]
  const float* logp_old;    // [R]
  double A, eps;
  double* loss_accum;       // device scalar, +=
  uint16_t* dlogits;        // bf16 [R, V]
  uint8_t* clip_mask;       // [R]
  float* logp_out;          // [R] or nullptr
  double* row_terms;        // workspace [R]
  uint32_t* status;
};
cudaError_t launch_grpo_loss(const LossArgs& a, cudaStream_t s);
// logp_out[t] = x_y - log sum_v exp(x_v) only (uses R, V, logits, ids, logp_out, status)
cudaError_t launch_token_logp(const LossArgs& a, cudaStream_t s);

// ----- elementwise helpers (k_elementwise.cu)
cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s);
cudaError_t launch_finalize(const float* acc, void* out, size_t n, float scale, int out_fp32,
                            int reset, cudaStream_t s);
cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t* status, cudaStream_t s);
// Context-parallel merge of n partial attention results (one per prompt shard) of rows x
// heads rows of D values: lse = log sum_r exp(lse_r), o = sum_r exp(lse_r - lse) o_r.
constexpr int kMaxParts = 16;
struct MergeArgs {
  int n;
  int64_t rows;               // R * Hq
  int D;
  const uint16_t* o_parts[kMaxParts];
  const float* lse_parts[kMaxParts];
  uint16_t* o;
  float* lse;
};
cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t s);
// out = bf16(sum_r float(parts_r)) over count elements (count a multiple of 8).
struct SumArgs {
  int n;
  int64_t count;
  const uint16_t* parts[kMaxParts];
  uint16_t* out;
};
cudaError_t launch_sum_bf16(const SumArgs& a, cudaStream_t s);
cudaError_t launch_scale_inplace(float* acc, size_t n, float scale, cudaStream_t s);
// Exact bf16 -> fp32 widening and fp32 -> bf16 rounding (nearest, ties to even) of count
// values (a multiple of 8, 16-byte aligned buffers).
cudaError_t launch_bf16_to_f32(const void* in, float* out, size_t count, cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float* in, void* out, size_t count, cudaStream_t s);

// ----- attention (k_attn_fwd.cu, k_attn_bwd.cu)
struct AttnShape {
  int64_t P, R;
  int Hq, Hkv, D, g;
  float scale;
  int qt;        // queries per 128-row tile (= 128 / g)
};

// Responses packed along the token axis: response b owns packed rows row0[b] .. row0[b+1]-1
// of Q/dO/O/dQ/LSE and of the suffix K/V, and sees the prompt and, causally, its own rows
// only (the shared-prefix tree).  One response is the case G = 1.  The prefix sums count
// each kernel's work units per response; a flat unit index maps to (response, local unit)
// with varlen_find.
constexpr int kMaxPacked = 64;
struct Varlen {
  int G;
  int row0[kMaxPacked + 1];   // packed row offsets; row0[G] = total rows
  int pair0[kMaxPacked + 1];  // forward units: pairs of 128-row Q tiles
  int qt0[kMaxPacked + 1];    // 128-row Q tiles
  int kt0[kMaxPacked + 1];    // 128-key suffix tiles
};

// The response b with pre[b] <= x < pre[b + 1] (pre non-decreasing, pre[0] = 0).
__host__ __device__ inline int varlen_find(const int* pre, int G, int x) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Fill v for G responses of lengths cu[b+1] - cu[b] (all >= 1) and qt queries per tile.
inline void varlen_build(Varlen* v, int G, const int64_t* cu, int qt) {
  v->G = G;
  v->row0[0] = v->pair0[0] = v->qt0[0] = v->kt0[0] = 0;
  for (int b = 0; b < G; ++b) {
    const int R = static_cast<int>(cu[b + 1] - cu[b]);
    const int nq = (R + qt - 1) / qt;
    v->row0[b + 1] = static_cast<int>(cu[b + 1]);
    v->pair0[b + 1] = v->pair0[b] + (nq + 1) / 2;
    v->qt0[b + 1] = v->qt0[b] + nq;
    v->kt0[b + 1] = v->kt0[b] + (R + 127) / 128;
  }
}

struct FwdArgs {
  AttnShape sh;               // sh.R = total packed rows
  Varlen vl;
  const CUtensorMap* tm_kp;   // prompt K [P][Hkv][D] 3-D map, box {64, 1, 128}
  const CUtensorMap* tm_vp;
  CUtensorMap tm_q;           // Q [R][Hq][D], box {64, g, qt}
  CUtensorMap tm_ks, tm_vs;   // suffix K/V [R][Hkv][D], box {64, 1, 128}
  uint16_t* o;
  float* lse;
  int no_suffix;              // 1: prompt keys only (one shard of a context-parallel prompt)
  uint32_t* status;
};
cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t s);

struct BwdArgs {
  AttnShape sh;               // sh.R = total packed rows
  Varlen vl;
  const CUtensorMap* tm_kp;   // prompt K/V [P][Hkv][D], box {64, 1, 128}
  const CUtensorMap* tm_vp;
  CUtensorMap tm_q, tm_do;    // [R][Hq][D], box {64, g, qt}
  CUtensorMap tm_ks, tm_vs;   // suffix K/V [R][Hkv][D], box {64, 1, 128}
  const float* rowstats;      // [Hkv][qt0[G]][256]: LSE log2 e of a tile's 128 rows, then Delta
  uint16_t* dq;               // bf16 [R, Hq, D]
  uint16_t* dk_suf;           // bf16 [R, Hkv, D] (unused when suffix_to_acc)
  uint16_t* dv_suf;
  float* dk_acc;              // fp32 [P, Hkv, D] (rows P .. P+R-1 too when suffix_to_acc)
  float* dv_acc;
  int suffix_to_acc;          // suffix key gradients are added into rows P + key of dk/dv_acc
  int no_suffix;              // 1: prompt keys only (one shard of a context-parallel prompt)
  uint32_t* status;
};
// Row statistics of every 128-row Q tile slot (kv, f, r) -- f the flat tile index over the
// packed responses, tile i = f - qt0[b] of response b, r = (t - i qt) g + h - kv g: valid
// rows get LSE log2 e and Delta = sum_d dO O; padding rows and rows past the response's
// end get (+inf, 0) so their softmax probabilities are exactly 0.
cudaError_t launch_bwd_prep(const uint16_t* o, const uint16_t* d_out, const float* lse,
                            float* rowstats, const AttnShape& sh, const Varlen& vl,
                            cudaStream_t s);
cudaError_t launch_attn_bwd_dkdv(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_attn_bwd_dq(const BwdArgs& a, cudaStream_t s);

int num_sms();
// Current device index for per-device host caches (launch attributes); -1 if unusable.
constexpr int kMaxDeviceCache = 64;
inline int cached_device_index() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDeviceCache) return -1;
  return dev;
}
// The per-thread message behind ls_last_error() (lives in ls_api.cu).
void set_last_error(const char* msg);
// The checks every handle-free entry point makes before it enqueues work: the current
// device is usable and `stream` (NULL = legacy default) belongs to it; *status receives the
// device's status word.  Returns an ls_status value.
int enter_call(void* stream, uint32_t** status);
// Records the CUDA message of a failed launch for ls_last_error(); returns LS_ERR_CUDA.
int launch_failed(cudaError_t e, const char* what);
// True when the launch attempt about to be made is the one ls_debug_fail_launch armed: the
// caller then skips the launch and reports a launch failure.
bool injected_failure();

}  // namespace ls
