// Fused GRPO clipped-surrogate loss (LongStraw review, section 1-1, equation L_policy).
//
// K5 grpo_loss_rows: one CTA per token row at a time (persistent over rows).
//   pass 1  streams the row's V bf16 logits with 128-bit loads and keeps a running
//           (max, sum of exp) pair: each 32-element group is summed as a fp32 tree and
//           added to a fp64 running sum; pairs combine across the CTA with warp shuffles.
//   chain   one thread runs the per-token scalar chain in fp64: lse, logp, rho, the clip
//           decision, the surrogate and g = d loss / d logp.
//   pass 2  re-reads the row (still in L2) and writes dlogits = g (onehot - softmax) in
//           bf16 with 128-bit streaming stores; a row with g == 0 (clipped, or A == 0)
//           is written as zeros without re-reading.
// K6 loss_reduce: one CTA sums the per-row loss terms in a fixed order (deterministic)
//           and adds the total into the fp64 loss accumulator.
// The scoring variant (old/reference-policy log-probs, review section 2-1 step 2) runs
// pass 1 and the log-prob only.
#include <cuda_bf16.h>

#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;                   // 4 x 8 = 32 logits per thread per step
constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLn2 = 0.69314718055994530942;

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
  x[0] = lo_bf16(v.x); x[1] = hi_bf16(v.x);
  x[2] = lo_bf16(v.y); x[3] = hi_bf16(v.y);
  x[4] = lo_bf16(v.z); x[5] = hi_bf16(v.z);
  x[6] = lo_bf16(v.w); x[7] = hi_bf16(v.w);
}

// Merge two (max, sum-of-exp relative to max) pairs; sums in fp64.  Max values are in
// log2 units (x * log2 e).
__device__ __forceinline__ void merge_ms(float& m, double& s, float m2, double s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) {
    s = s * static_cast<double>(ex2_approx(m - m2)) + s2;
    m = m2;
  } else {
    s += s2 * static_cast<double>(ex2_approx(m2 - m));
  }
}

// kScore: log-prob only (old/reference-policy scoring): pass 1 and logp, no loss, no
// dlogits, no second read of the row.
template <bool kVec, bool kScore>
__global__ void __launch_bounds__(kThreads) grpo_loss_rows(LossArgs a) {
  __shared__ float sh_m[kThreads / 32];
  __shared__ double sh_s[kThreads / 32];
  __shared__ float sh_g, sh_lse2;
  __shared__ int sh_y;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;

  for (int64_t row = blockIdx.x; row < a.R; row += gridDim.x) {
    const uint16_t* xr = a.logits + row * V;

    // ---------------- pass 1: running max (log2 units) and sum of exp2
    float m = -INFINITY;
    double s = 0.0;
    if (kVec) {
      const uint4* x4 = reinterpret_cast<const uint4*>(xr);
      const int64_t nvec = V >> 3;
      for (int64_t base = tid; base < nvec; base += kThreads * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t i = base + static_cast<int64_t>(u) * kThreads;
          v[u] = (i < nvec) ? __ldg(x4 + i) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
        float x[kUnroll][8];
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          unpack8(v[u], x[u]);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            x[u][k] *= kLog2e;
            cm = fmaxf(cm, x[u][k]);
          }
        }
        if (cm == -INFINITY) continue;
        if (cm > m) {
          if (m != -INFINITY) s *= static_cast<double>(ex2_approx(m - cm));
          m = cm;
        }
        float cs[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          float e[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) e[k] = ex2_approx(x[u][k] - m);
          cs[u] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
        }
        s += static_cast<double>((cs[0] + cs[1]) + (cs[2] + cs[3]));
      }
    } else {
      for (int64_t i = tid; i < V; i += kThreads) {
        const float x = __uint_as_float(static_cast<uint32_t>(xr[i]) << 16) * kLog2e;
        if (x > m) {
          if (m != -INFINITY) s *= static_cast<double>(ex2_approx(m - x));
          m = x;
        }
        s += static_cast<double>(ex2_approx(x - m));
      }
    }
    // CTA-wide merge of (m, s)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const double s2 = __shfl_xor_sync(0xffffffffu, s, off);
      merge_ms(m, s, m2, s2);
    }
    if (lane == 0) { sh_m[warp] = m; sh_s[warp] = s; }
    __syncthreads();

    // ---------------- per-token scalar chain (fp64), one thread
    if (tid == 0) {
      float M = sh_m[0];
      double S = sh_s[0];
      for (int w = 1; w < kThreads / 32; ++w) merge_ms(M, S, sh_m[w], sh_s[w]);
      const int32_t y = a.ids[row];
      if constexpr (kScore) {
        double lp = 0.0;
        if (y < 0 || y >= V) {
          set_device_status(a.status, DEV_BAD_INDEX);
        } else {
          const double lse = (static_cast<double>(M) + log2(S)) * kLn2;
          lp = static_cast<double>(__uint_as_float(static_cast<uint32_t>(xr[y]) << 16)) - lse;
        }
        a.logp_out[row] = static_cast<float>(lp);
      } else {
        const double GR = static_cast<double>(a.G) * static_cast<double>(a.R);
        double term = 0.0, g = 0.0, lse = 0.0, logp = 0.0;
        uint8_t clipped = 0;
        if (y < 0 || y >= V) {
          set_device_status(a.status, DEV_BAD_INDEX);
          logp = 0.0;
          lse = 0.0;
        } else {
          // lse in natural log: (M + log2 S) * ln 2
          lse = (static_cast<double>(M) + log2(S)) * kLn2;
          const double xy = static_cast<double>(__uint_as_float(static_cast<uint32_t>(xr[y]) << 16));
          logp = xy - lse;
          const double rho = exp(logp - static_cast<double>(a.logp_old[row]));
          const double A = a.A;
          const double clo = 1.0 - a.eps, chi = 1.0 + a.eps;
          const double rclip = rho < clo ? clo : (rho > chi ? chi : rho);
          const double unclipped_val = rho * A;
          const double clipped_val = rclip * A;
          clipped = (clipped_val < unclipped_val) ? 1 : 0;
          const double surr = clipped ? clipped_val : unclipped_val;
          term = -surr / GR;
          g = clipped ? 0.0 : -A * rho / GR;
        }
        a.row_terms[row] = term;
        a.clip_mask[row] = clipped;
        if (a.logp_out != nullptr) a.logp_out[row] = static_cast<float>(logp);
        sh_g = static_cast<float>(g);
        sh_lse2 = static_cast<float>(lse / kLn2);    // lse in log2 units
        sh_y = (y < 0 || y >= V) ? -1 : y;
      }
    }
    __syncthreads();
    if constexpr (kScore) continue;
    const float g = sh_g, lse2 = sh_lse2;
    const int y = sh_y;

    // ---------------- pass 2: dlogits = g * (onehot - softmax)
    uint16_t* dr = a.dlogits + row * V;
    if (kVec) {
      uint4* d4 = reinterpret_cast<uint4*>(dr);
      const uint4* x4 = reinterpret_cast<const uint4*>(xr);
      const int64_t nvec = V >> 3;
      if (g == 0.0f) {
        for (int64_t i = tid; i < nvec; i += kThreads) __stcs(d4 + i, make_uint4(0u, 0u, 0u, 0u));
      } else {
        for (int64_t base = tid; base < nvec; base += kThreads * kUnroll) {
          uint4 v[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * kThreads;
            if (i < nvec) v[u] = __ldcs(x4 + i);
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * kThreads;
            if (i < nvec) {
              float x[8];
              unpack8(v[u], x);
              float d[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float p = ex2_approx(fmaf(x[k], kLog2e, -lse2));
                const float oh = (i * 8 + k == y) ? 1.0f : 0.0f;
                d[k] = g * (oh - p);
              }
              uint4 o;
              o.x = pack_bf16x2(d[0], d[1]);
              o.y = pack_bf16x2(d[2], d[3]);
              o.z = pack_bf16x2(d[4], d[5]);
              o.w = pack_bf16x2(d[6], d[7]);
              __stcs(d4 + i, o);
            }
          }
        }
      }
    } else {
      for (int64_t i = tid; i < V; i += kThreads) {
        float d = 0.0f;
        if (g != 0.0f) {
          const float x = __uint_as_float(static_cast<uint32_t>(xr[i]) << 16);
          const float p = ex2_approx(fmaf(x, kLog2e, -lse2));
          d = g * (((i == y) ? 1.0f : 0.0f) - p);
        }
        __nv_bfloat16 b = __float2bfloat16_rn(d);
        dr[i] = *reinterpret_cast<uint16_t*>(&b);
      }
    }
    __syncthreads();   // shared scalars are rewritten by the next row
  }
}

constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads) loss_reduce(const double* terms, int64_t n,
                                                             double* loss_accum) {
  __shared__ double sh[kReduceThreads];
  const int tid = threadIdx.x;
  double acc = 0.0;
  for (int64_t i = tid; i < n; i += kReduceThreads) acc += terms[i];
  sh[tid] = acc;
  __syncthreads();
  for (int w = kReduceThreads / 2; w > 0; w >>= 1) {
    if (tid < w) sh[tid] += sh[tid + w];
    __syncthreads();
  }
  if (tid == 0) *loss_accum += sh[0];
}

}  // namespace

cudaError_t launch_grpo_loss(const LossArgs& a, cudaStream_t s) {
  const bool vec = (a.V % 8 == 0) && (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.dlogits) % 16 == 0);
  int64_t grid = static_cast<int64_t>(num_sms()) * 4;
  if (grid > a.R) grid = a.R;
  if (vec)
    grpo_loss_rows<true, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
  else
    grpo_loss_rows<false, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  loss_reduce<<<1, kReduceThreads, 0, s>>>(a.row_terms, a.R, a.loss_accum);
  return cudaGetLastError();
}

cudaError_t launch_token_logp(const LossArgs& a, cudaStream_t s) {
  const bool vec = (a.V % 8 == 0) && (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0);
  int64_t grid = static_cast<int64_t>(num_sms()) * 4;
  if (grid > a.R) grid = a.R;
  if (vec)
    grpo_loss_rows<true, true><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
  else
    grpo_loss_rows<false, true><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ls
