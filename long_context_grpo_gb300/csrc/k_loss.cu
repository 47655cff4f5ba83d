// Fused GRPO clipped-surrogate loss (LongStraw review, section 1-1, equation L_policy).
//
// K5 grpo_loss_cluster (V a multiple of 8, 16-byte aligned rows): a cluster of 4 CTAs owns
//   one token row at a time and CTA c streams the c-th quarter of it, so the rows in flight
//   (about 150 at once) stay small enough for the second read to come from L2.
//   pass 1  8 streaming warps keep a running (max, compensated fp32 sum of exp2) per thread
//           (TwoSum: no fp64 on the streaming path), merged across the warp.
//   scalar  a ninth warp merges the CTA's partials, sends them to the other three CTAs
//           through distributed shared memory with a remote mbarrier arrive (bounded wait),
//           merges the four in rank order (the same result in every CTA), assembles lse in
//           fp64 from an exponent/mantissa split, and decides the clip and g from rho in
//           fp32; after releasing the streaming warps it computes the row's loss term in
//           fp64 (CTA 0 writes the row's outputs).
//   pass 2  the streaming warps re-read their quarter (L2) and write dlogits = g (onehot -
//           softmax) in bf16 with streaming stores.
//   Scoring (log-prob only) prefetches the next row's quarter into L2 with a bulk prefetch.
// K5 grpo_loss_rows (any V): one CTA per token row at a time; the same steps with the row
//   streamed from global memory twice (the second read mostly from L2).
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


// ======================================================================================
// K5, cluster version
// ======================================================================================
constexpr int kCl = 4;                       // CTAs per row (one cluster)
constexpr int kCThreads = 256;               // streaming threads per CTA
constexpr int kCWarps = kCThreads / 32;
constexpr int kClThreads = kCThreads + 32;   // + the scalar warp
constexpr int kCUnroll = 4;                  // 4 x 8 = 32 logits per thread per step

// hi + lo += t, with the exact error of the fp32 addition kept in lo (TwoSum).
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float t) {
  const float s = hi + t;
  const float bp = s - hi;
  const float err = (hi - (s - bp)) + (t - bp);
  hi = s;
  lo += err;
}

// Merge the partial (m2, h2 + l2) into (m, h + l): sums of exp2(x log2 e - m), max m in
// log2 units; the smaller-max side is rescaled by exp2 of the difference.
__device__ __forceinline__ void ms_merge(float& m, float& h, float& l, float m2, float h2, float l2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; h = h2; l = l2; return; }
  if (m2 > m) {
    const float f = ex2_approx(m - m2);
    h *= f; l *= f; m = m2;
  } else {
    const float f = ex2_approx(m2 - m);
    h2 *= f; l2 *= f;
  }
  l += l2;
  two_sum_acc(h, l, h2);
}

// Pass 1 over this CTA's slice of one row: running (max, compensated sum of exp2), merged
// across the warp; lane 0 of each warp leaves (m, hi, lo) in part[warp].
__device__ __forceinline__ void slice_pass1(const uint4* x4, int nvec, int tid, float (*part)[3]) {
  float m = -INFINITY, hi = 0.0f, lo = 0.0f;
  for (int base = tid; base < nvec; base += kCThreads * kCUnroll) {
    uint4 v[kCUnroll];
#pragma unroll
    for (int u = 0; u < kCUnroll; ++u) {
      const int i = base + u * kCThreads;
      v[u] = (i < nvec) ? __ldg(x4 + i) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
    float x[kCUnroll][8];
    float cm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kCUnroll; ++u) {
      unpack8(v[u], x[u]);
#pragma unroll
      for (int k = 0; k < 8; ++k) cm = fmaxf(cm, x[u][k]);
    }
    if (cm == -INFINITY) continue;
    const float cm2 = cm * kLog2e;
    if (cm2 > m) {
      if (m != -INFINITY) {
        const float f = ex2_approx(m - cm2);
        hi *= f; lo *= f;
      }
      m = cm2;
    }
    float cs[kCUnroll];
#pragma unroll
    for (int u = 0; u < kCUnroll; ++u) {
      float e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = ex2_approx(fmaf(x[u][k], kLog2e, -m));
      cs[u] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    }
    two_sum_acc(hi, lo, (cs[0] + cs[1]) + (cs[2] + cs[3]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, off);
    ms_merge(m, hi, lo, m2, h2, l2);
  }
  if ((tid & 31) == 0) {
    const int w = tid >> 5;
    part[w][0] = m; part[w][1] = hi; part[w][2] = lo;
  }
  __threadfence_block();
  __syncwarp();
}

// Named barriers (id 0 is __syncthreads): partials of row k ready -> kBarParts + (k & 1);
// g of row k ready -> kBarG + (k & 1).  Alternating ids and buffers keep consecutive rows
// apart while the scalar warp finishes the previous row's loss term.
enum : uint32_t { kBarParts = 1, kBarG = 3 };
__device__ __forceinline__ void bar_sync_par(uint32_t base, uint32_t par) {
  if (par) named_barrier_sync(base + 1, kClThreads); else named_barrier_sync(base, kClThreads);
}
__device__ __forceinline__ void bar_arrive_par(uint32_t base, uint32_t par) {
  if (par) named_barrier_arrive(base + 1, kClThreads); else named_barrier_arrive(base, kClThreads);
}

template <bool kScore>
__global__ void __launch_bounds__(kClThreads, 4) grpo_loss_cluster(LossArgs a, int64_t vc, float gscale) {
  __shared__ __align__(8) uint64_t xbar[2];      // 4 arrivals per row (row parity): partials in
  __shared__ float part[2][kCWarps][3];          // per streaming warp: (m, hi, lo), row parity
  __shared__ float slot[2][kCl][3];              // per rank, row parity
  __shared__ float sh_g[2], sh_lse2[2];
  __shared__ int sh_yl[2];
  // Set to 1 when a bounded wait of this CTA or of a peer gave up: from then on no CTA of
  // the cluster exchanges partials any more, rows are only walked through (same barrier
  // sequence, no loads) and their loss terms and log-probs are written as NaN.
  __shared__ int cl_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int64_t V = a.V, R = a.R;
  const int64_t c0 = static_cast<int64_t>(rank) * vc;
  int64_t clen = V - c0;
  clen = clen < 0 ? 0 : (clen > vc ? vc : clen);
  const int nvec = static_cast<int>(clen >> 3);

  if (tid == 0) {
    cl_abort = 0;
    mbar_init(&xbar[0], kCl);
    mbar_init(&xbar[1], kCl);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();   // peers' barriers are initialised before any remote arrive

  const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
  volatile int* vabort = &cl_abort;

  if (warp == kCWarps) {
    // ------------------------------------------------------------------ scalar warp
    int it = 0;
    for (int64_t row = cid; row < R; row += ncl, ++it) {
      const uint32_t par = static_cast<uint32_t>(it & 1);
      // row inputs fetched before the partials arrive
      int32_t y = 0;
      float old = 0.0f, xy = 0.0f;
      if (lane == 0) {
        // scoring: the next row's slice streams into L2 while this row is processed (the
        // loss keeps L2 for its second read of the current row instead)
        if (kScore && row + ncl < R && nvec > 0)
          bulk_prefetch_l2(a.logits + (row + ncl) * V + c0, static_cast<uint32_t>(nvec) * 16u);
        y = a.ids[row];
        if (!kScore) old = a.logp_old[row];
        if (y >= 0 && y < V) xy = __uint_as_float(static_cast<uint32_t>(__ldg(a.logits + row * V + y)) << 16);
      }
      bar_sync_par(kBarParts, par);
      float m = -INFINITY, h = 0.0f, l = 0.0f;
      if (lane < kCWarps) { m = part[par][lane][0]; h = part[par][lane][1]; l = part[par][lane][2]; }
      if (kScore) bar_arrive_par(kBarG, par);   // part[par] may be rewritten
#pragma unroll
      for (int off = kCWarps / 2; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float h2 = __shfl_xor_sync(0xffffffffu, h, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        ms_merge(m, h, l, m2, h2, l2);
      }
      // lane 0: exchange, lse, and (loss) the clip decision and g
      bool bad = false, clipped = false, aborted = false;
      double logp = 0.0, dl = 0.0;
      if (lane == 0) {
        aborted = *vabort != 0;
        if (!aborted) {
#pragma unroll
          for (int r = 0; r < kCl; ++r) {
            const uint32_t dst = cluster_map(&slot[par][rank][0], r);
            st_cluster_f32(dst, m);
            st_cluster_f32(dst + 4, h);
            st_cluster_f32(dst + 8, l);
          }
          // xbar[par] completes one phase every second row
#pragma unroll
          for (int r = 0; r < kCl; ++r) mbar_arrive_remote(cluster_map(&xbar[par], r));
          aborted = !mbar_wait_cluster(&xbar[par], static_cast<uint32_t>((it >> 1) & 1), a.status,
                                       vabort);
          // a wait that gave up stops the exchange in every CTA of the cluster (the peers'
          // own waits poll the flag); the CTAs stay resident until the final cluster barrier
          if (aborted) {
#pragma unroll
            for (int r = 0; r < kCl; ++r) st_cluster_u32(cluster_map(&cl_abort, r), 1u);
          }
        }
      }
      aborted = __shfl_sync(0xffffffffu, aborted ? 1 : 0, 0) != 0;
      if (aborted) {
        if (lane == 0) {
          if constexpr (kScore) {
            if (rank == 0) a.logp_out[row] = __int_as_float(0x7fc00000);
          } else {
            sh_g[par] = 0.0f;
            sh_lse2[par] = 0.0f;
            sh_yl[par] = -1;
            __threadfence_block();
          }
        }
        __syncwarp();
        if constexpr (!kScore) {
          bar_arrive_par(kBarG, par);
          if (lane == 0 && rank == 0) {
            const double nan = __longlong_as_double(0x7ff8000000000000ll);
            a.row_terms[row] = nan;
            a.clip_mask[row] = 0;
            if (a.logp_out != nullptr) a.logp_out[row] = __int_as_float(0x7fc00000);
          }
        }
        __syncwarp();
        continue;
      }
      if (lane == 0) {
        // the row's partials in rank order: the same result in every CTA of the cluster
        float M = slot[par][0][0], H = slot[par][0][1], L = slot[par][0][2];
#pragma unroll
        for (int r = 1; r < kCl; ++r) ms_merge(M, H, L, slot[par][r][0], slot[par][r][1], slot[par][r][2]);
        // lse in log2 units = M + log2(H + L): exponent and mantissa of H taken apart so the
        // fp32 log2 only sees [0.5, 1); assembled in fp64.
        int e2 = 0;
        const float mant = frexpf(H, &e2);
        const float corr = (L / H) * 1.4426950408889634f;
        const double lse2 = static_cast<double>(M) +
                            (static_cast<double>(e2) + (static_cast<double>(log2f(mant)) + static_cast<double>(corr)));
        bad = (y < 0 || y >= V);
        logp = bad ? 0.0 : static_cast<double>(xy) - lse2 * kLn2;
        if constexpr (kScore) {
          if (rank == 0) {
            if (bad) set_device_status(a.status, DEV_BAD_INDEX);
            a.logp_out[row] = static_cast<float>(logp);
          }
        } else {
          // rho in fp32 from the fp64 log-ratio decides the clip and g
          dl = logp - static_cast<double>(old);
          const float rho_f = expf(static_cast<float>(dl));
          const double rho_d32 = static_cast<double>(rho_f);
          clipped = !bad && ((a.A > 0.0 && rho_d32 > 1.0 + a.eps) || (a.A < 0.0 && rho_d32 < 1.0 - a.eps));
          sh_g[par] = (bad || clipped) ? 0.0f : gscale * rho_f;
          sh_lse2[par] = static_cast<float>(lse2);
          sh_yl[par] = (bad || y - c0 < 0 || y - c0 >= clen) ? -1 : static_cast<int>(y - c0);
          __threadfence_block();
        }
      }
      __syncwarp();
      if constexpr (!kScore) {
        bar_arrive_par(kBarG, par);
        // after the streaming warps are released: the row's loss term in fp64 (CTA 0)
        if (lane == 0 && rank == 0) {
          double term = 0.0;
          if (bad) {
            set_device_status(a.status, DEV_BAD_INDEX);
          } else {
            const double A = a.A;
            const double rho = exp(dl);
            const double clo = 1.0 - a.eps, chi = 1.0 + a.eps;
            const double rclip = rho < clo ? clo : (rho > chi ? chi : rho);
            const double surr = clipped ? rclip * A : rho * A;
            term = -surr / (static_cast<double>(a.G) * static_cast<double>(a.R));
          }
          a.row_terms[row] = term;
          a.clip_mask[row] = clipped ? 1 : 0;
          if (a.logp_out != nullptr) a.logp_out[row] = static_cast<float>(logp);
        }
      }
      __syncwarp();
    }
  } else {
    // -------------------------------------------------------------- streaming warps
    int it = 0;
    for (int64_t row = cid; row < R; row += ncl, ++it) {
      const uint32_t par = static_cast<uint32_t>(it & 1);
      if (!*vabort)
        slice_pass1(reinterpret_cast<const uint4*>(a.logits + row * V + c0), nvec, tid, part[par]);
      bar_arrive_par(kBarParts, par);
      bar_sync_par(kBarG, par);
      if constexpr (kScore) continue;

      // pass 2: dlogits = g (onehot - softmax), the slice re-read from L2
      const float g = sh_g[par], lse2 = sh_lse2[par];
      const int yl = sh_yl[par];
      const uint4* x4 = reinterpret_cast<const uint4*>(a.logits + row * V + c0);
      uint4* d4 = reinterpret_cast<uint4*>(a.dlogits + row * V + c0);
      if (g == 0.0f) {
        for (int i = tid; i < nvec; i += kCThreads) __stcs(d4 + i, make_uint4(0u, 0u, 0u, 0u));
      } else {
        const float ng = -g;
        for (int base = tid; base < nvec; base += kCThreads * kCUnroll) {
          uint4 v[kCUnroll];
#pragma unroll
          for (int u = 0; u < kCUnroll; ++u) {
            const int i = base + u * kCThreads;
            if (i < nvec) v[u] = __ldcs(x4 + i);
          }
#pragma unroll
          for (int u = 0; u < kCUnroll; ++u) {
            const int i = base + u * kCThreads;
            if (i < nvec) {
              const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
              uint32_t o[4];
              const int rel = yl - i * 8;   // one-hot position in this vector
              if (static_cast<unsigned>(rel) < 8u) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float pa = ex2_approx(fmaf(lo_bf16(w[q]), kLog2e, -lse2));
                  const float pb = ex2_approx(fmaf(hi_bf16(w[q]), kLog2e, -lse2));
                  o[q] = pack_bf16x2(g * ((2 * q == rel ? 1.0f : 0.0f) - pa),
                                     g * ((2 * q + 1 == rel ? 1.0f : 0.0f) - pb));
                }
              } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float pa = ex2_approx(fmaf(lo_bf16(w[q]), kLog2e, -lse2));
                  const float pb = ex2_approx(fmaf(hi_bf16(w[q]), kLog2e, -lse2));
                  o[q] = pack_bf16x2(ng * pa, ng * pb);
                }
              }
              __stcs(d4 + i, make_uint4(o[0], o[1], o[2], o[3]));
            }
          }
        }
      }
    }
  }
  __syncwarp();
  // No CTA leaves while a peer may still write its shared memory.  Every wait before this
  // point is bounded (and after an abort no CTA waits on a peer any more), so every thread
  // of the cluster reaches this barrier in bounded time.
  cluster_sync_all();
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

// Slice length (elements, a multiple of 8) of each CTA of the cluster kernel, or 0 when
// the row layout does not allow it (V not a multiple of 8, unaligned rows, tiny or huge V).
static int64_t cluster_slice(const LossArgs& a, bool with_dlogits) {
  if (a.V % 8 != 0 || a.V < 8 * kCl) return 0;
  if (reinterpret_cast<uintptr_t>(a.logits) % 16 != 0) return 0;
  if (with_dlogits && reinterpret_cast<uintptr_t>(a.dlogits) % 16 != 0) return 0;
  const int64_t vc = ((a.V + kCl - 1) / kCl + 7) / 8 * 8;
  return vc;
}

template <bool kScore>
static cudaError_t launch_cluster(const LossArgs& a, int64_t vc, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms()) * 4u, 1, 1);
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, grpo_loss_cluster<kScore>, &cfg) != cudaSuccess ||
      nclusters <= 0) {
    (void)cudaGetLastError();
    nclusters = num_sms() / kCl;
  }
  if (nclusters > a.R) nclusters = static_cast<int>(a.R);
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * kCl), 1, 1);
  const float gscale = static_cast<float>(-a.A / (static_cast<double>(a.G) * static_cast<double>(a.R)));
  return cudaLaunchKernelEx(&cfg, grpo_loss_cluster<kScore>, a, vc, gscale);
}

cudaError_t launch_grpo_loss(const LossArgs& a, cudaStream_t s) {
  cudaError_t e;
  const int64_t vc = cluster_slice(a, true);
  if (vc > 0) {
    e = launch_cluster<false>(a, vc, s);
  } else {
    const bool vec = (a.V % 8 == 0) && (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.dlogits) % 16 == 0);
    int64_t grid = static_cast<int64_t>(num_sms()) * 4;
    if (grid > a.R) grid = a.R;
    if (vec)
      grpo_loss_rows<true, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
    else
      grpo_loss_rows<false, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  loss_reduce<<<1, kReduceThreads, 0, s>>>(a.row_terms, a.R, a.loss_accum);
  return cudaGetLastError();
}

cudaError_t launch_token_logp(const LossArgs& a, cudaStream_t s) {
  const int64_t vc = cluster_slice(a, false);
  if (vc > 0) return launch_cluster<true>(a, vc, s);
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
