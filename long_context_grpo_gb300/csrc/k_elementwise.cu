// Bandwidth kernels around the replay:
//   K0 zero_f32        zero the fp32 prompt-gradient accumulators (prompt capture hand-off)
//   K7 finalize        out = scale * acc (bf16 or fp32), optionally zeroing acc: the group's
//                      one finalization (LongStraw review, section 2-1 step 5)
//   K2 bwd_prep        Delta[t,h] = sum_d dO[t,h,d] O[t,h,d], the row term of the softmax
//                      backward dS = P * (dP - Delta), packed with LSE by 128-row Q tile
//   merge              context-parallel combination of per-shard partial attention results:
//                      lse = log sum_r exp(lse_r), o = sum_r exp(lse_r - lse) o_r
//                      (LongStraw review, section 3-2 (2): global LSE/output merge)
//   sum_bf16           sum of per-shard dQ partials, fp32 accumulation, bf16 out
//   bf16 <-> f32       conversions around the cross-rank fp32 sum of the dQ parts
// All use 128-bit accesses on a grid sized to the SM count.
#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) zero_f32_kernel(float4* p, size_t n4, float* tail,
                                                           size_t ntail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n4; i += stride)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = 0.f;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads) finalize_kernel(float4* acc, void* out, size_t n4,
                                                           float scale, int reset) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n4; i += stride) {
    float4 a = __ldcs(acc + i);
    a.x *= scale; a.y *= scale; a.z *= scale; a.w *= scale;
    if (kOutF32) {
      __stcs(reinterpret_cast<float4*>(out) + i, a);
    } else {
      uint2 b;
      b.x = bf16x2_rn(a.x, a.y);
      b.y = bf16x2_rn(a.z, a.w);
      __stcs(reinterpret_cast<uint2*>(out) + i, b);
    }
    if (reset) __stcs(acc + i, make_float4(0.f, 0.f, 0.f, 0.f));
  }
}

__global__ void __launch_bounds__(kThreads) scale_kernel(float4* acc, size_t n4, float scale) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n4; i += stride) {
    float4 a = acc[i];
    a.x *= scale; a.y *= scale; a.z *= scale; a.w *= scale;
    acc[i] = a;
  }
}

// One warp per 128-row Q tile slot (kv, i, r): row r of tile i packs query
// t = i * qt + r / g and head h = kv * g + r % g.  Valid rows get LSE log2 e and
// Delta = sum_d dO O; padding rows and rows past R get (+inf, 0).  Layout per tile: the
// 128 LSE values, then the 128 Delta values.
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(const uint4* o, const uint4* d_out,
                                                           const float* lse, float* rowstats,
                                                           AttnShape sh,
                                                           const __grid_constant__ Varlen vl) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const int per_row = sh.D / 8;   // 8 or 16 lanes, 8 bf16 each
  const int64_t n_qt = vl.qt0[vl.G];
  const int64_t slots = static_cast<int64_t>(sh.Hkv) * n_qt * 128;
  for (int64_t sidx = blockIdx.x * static_cast<int64_t>(kThreads / 32) + (threadIdx.x >> 5);
       sidx < slots; sidx += warps_total) {
    const int64_t tile = sidx >> 7;                // kv * n_qt + f
    const int r = static_cast<int>(sidx & 127);
    const int64_t kv = tile / n_qt;
    const int f = static_cast<int>(tile - kv * n_qt);
    const int b = varlen_find(vl.qt0, vl.G, f);
    const int64_t t = static_cast<int64_t>(f - vl.qt0[b]) * sh.qt + r / sh.g;
    const int64_t h = kv * sh.g + r % sh.g;
    const bool valid = (r < sh.g * sh.qt) && (t < vl.row0[b + 1] - vl.row0[b]);
    const int64_t row = (vl.row0[b] + t) * sh.Hq + h;
    float acc = 0.f;
    if (valid && lane < per_row) {
      const uint4 a = __ldcs(o + row * per_row + lane);
      const uint4 bb = __ldcs(d_out + row * per_row + lane);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), acc);
        acc = fmaf(__uint_as_float(aw[k] & 0xFFFF0000u), __uint_as_float(bw[k] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      float* dst = rowstats + tile * 256;
      dst[r] = valid ? lse[row] * 1.4426950408889634f : INFINITY;
      dst[128 + r] = valid ? acc : 0.f;
    }
  }
}

// One thread per (row, 8 output values).  The shard weights exp(lse_r - m) are recomputed
// per shard instead of kept in an array, so nothing is indexed dynamically.
__global__ void __launch_bounds__(kThreads) attn_merge_kernel(const __grid_constant__ MergeArgs a) {
  const int per_row = a.D / 8;
  const int64_t total = a.rows * per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t row = idx / per_row;
    const int c = static_cast<int>(idx - row * per_row);
    float m = -INFINITY;
    for (int r = 0; r < a.n; ++r) m = fmaxf(m, a.lse_parts[r][row]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float ssum = 0.f;
    if (m != -INFINITY) {
      for (int r = 0; r < a.n; ++r) ssum += expf(a.lse_parts[r][row] - m);
      const float inv = 1.0f / ssum;
      for (int r = 0; r < a.n; ++r) {
        const float wr = expf(a.lse_parts[r][row] - m) * inv;
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(a.o_parts[r] + row * a.D) + c);
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] = fmaf(wr, __uint_as_float(vw[k] << 16), acc[2 * k]);
          acc[2 * k + 1] = fmaf(wr, __uint_as_float(vw[k] & 0xFFFF0000u), acc[2 * k + 1]);
        }
      }
    }
    uint4 o;
    o.x = bf16x2_rn(acc[0], acc[1]);
    o.y = bf16x2_rn(acc[2], acc[3]);
    o.z = bf16x2_rn(acc[4], acc[5]);
    o.w = bf16x2_rn(acc[6], acc[7]);
    __stcs(reinterpret_cast<uint4*>(a.o + row * a.D) + c, o);
    if (c == 0) a.lse[row] = (m == -INFINITY) ? -INFINITY : m + logf(ssum);
  }
}

__global__ void __launch_bounds__(kThreads) sum_bf16_kernel(const __grid_constant__ SumArgs a) {
  const int64_t n8 = a.count / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n8; i += stride) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < a.n; ++r) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(a.parts[r]) + i);
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] += __uint_as_float(vw[k] << 16);
        acc[2 * k + 1] += __uint_as_float(vw[k] & 0xFFFF0000u);
      }
    }
    uint4 o;
    o.x = bf16x2_rn(acc[0], acc[1]);
    o.y = bf16x2_rn(acc[2], acc[3]);
    o.z = bf16x2_rn(acc[4], acc[5]);
    o.w = bf16x2_rn(acc[6], acc[7]);
    __stcs(reinterpret_cast<uint4*>(a.out) + i, o);
  }
}

// Element-type conversions of the context-parallel dQ exchange: the bf16 dQ part of a
// shard is summed across ranks in fp32 (8 values per thread, 128-bit accesses).
__global__ void __launch_bounds__(kThreads) bf16_to_f32_kernel(const uint4* in, float4* out,
                                                              size_t n8) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n8; i += stride) {
    const uint4 v = __ldcs(in + i);
    __stcs(out + 2 * i, make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                    __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)));
    __stcs(out + 2 * i + 1, make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                        __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)));
  }
}

__global__ void __launch_bounds__(kThreads) f32_to_bf16_kernel(const float4* in, uint4* out,
                                                              size_t n8) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n8; i += stride) {
    const float4 a = __ldcs(in + 2 * i), b = __ldcs(in + 2 * i + 1);
    uint4 o;
    o.x = bf16x2_rn(a.x, a.y);
    o.y = bf16x2_rn(a.z, a.w);
    o.z = bf16x2_rn(b.x, b.y);
    o.w = bf16x2_rn(b.z, b.w);
    __stcs(out + i, o);
  }
}

// Failure-detection self test: one thread waits on an mbarrier that nothing arrives at,
// bounded by limit_ns, then records DEV_WAIT_TIMEOUT exactly as the replay kernels do when
// a wait gives up, and exits; the context stays usable.
__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_ns(&bar, 0u, limit_ns)) set_device_status(status, DEV_WAIT_TIMEOUT);
  }
}

unsigned grid_for(size_t work_items) {
  const size_t per_block = kThreads;
  size_t blocks = (work_items + per_block - 1) / per_block;
  const size_t cap = static_cast<size_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s) {
  const size_t n4 = n / 4, ntail = n % 4;
  zero_f32_kernel<<<grid_for(n4), kThreads, 0, s>>>(reinterpret_cast<float4*>(p), n4,
                                                     p + n4 * 4, ntail);
  return cudaGetLastError();
}

// n is a multiple of 4 (P * Hkv * D with D in {64, 128}).
cudaError_t launch_finalize(const float* acc, void* out, size_t n, float scale, int out_fp32,
                            int reset, cudaStream_t s) {
  const size_t n4 = n / 4;
  float4* a4 = reinterpret_cast<float4*>(const_cast<float*>(acc));
  if (out_fp32)
    finalize_kernel<true><<<grid_for(n4), kThreads, 0, s>>>(a4, out, n4, scale, reset);
  else
    finalize_kernel<false><<<grid_for(n4), kThreads, 0, s>>>(a4, out, n4, scale, reset);
  return cudaGetLastError();
}

cudaError_t launch_scale_inplace(float* acc, size_t n, float scale, cudaStream_t s) {
  const size_t n4 = n / 4;
  scale_kernel<<<grid_for(n4), kThreads, 0, s>>>(reinterpret_cast<float4*>(acc), n4, scale);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t* status, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t s) {
  attn_merge_kernel<<<grid_for(static_cast<size_t>(a.rows) * (a.D / 8)), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sum_bf16(const SumArgs& a, cudaStream_t s) {
  sum_bf16_kernel<<<grid_for(static_cast<size_t>(a.count / 8)), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f32(const void* in, float* out, size_t count, cudaStream_t s) {
  bf16_to_f32_kernel<<<grid_for(count / 8), kThreads, 0, s>>>(static_cast<const uint4*>(in),
                                                             reinterpret_cast<float4*>(out), count / 8);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* in, void* out, size_t count, cudaStream_t s) {
  f32_to_bf16_kernel<<<grid_for(count / 8), kThreads, 0, s>>>(reinterpret_cast<const float4*>(in),
                                                             static_cast<uint4*>(out), count / 8);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const uint16_t* o, const uint16_t* d_out, const float* lse,
                            float* rowstats, const AttnShape& sh, const Varlen& vl,
                            cudaStream_t s) {
  const size_t slots = static_cast<size_t>(sh.Hkv) * vl.qt0[vl.G] * 128;
  bwd_prep_kernel<<<grid_for(slots * 32), kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(d_out), lse, rowstats, sh,
      vl);
  return cudaGetLastError();
}

}  // namespace ls
