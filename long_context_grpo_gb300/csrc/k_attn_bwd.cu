// Backward replay of one response (LongStraw review, dimensionstp.github.io "LongStraw",
// section 2-1 step 4: the suffix graph is released after its backward and only gradients
// are accumulated; section 2-2: the prompt-side gradient at the boundary state z_P, which
// for one attention layer is d loss / d (prompt K, V)).
//
// With P = exp(s Q K^T - LSE) (recomputed from the forward's LSE), dP = dO V^T,
// Delta = rowsum(dO * O) and dS = P * (dP - Delta):
//   dV = P^T dO,  dK = s dS^T Q,  dQ = s dS K.
//
// K3 attn_bwd_dkdv (key-tile outer): a work unit is one 128-key tile of one kv head, either
//   a prompt tile or a suffix tile.  The unit sweeps every 64-row Q/dO sub-tile that sees
//   its keys (qt64 = 64/g queries x g heads), computing S^T = K Q^T and dP^T = V dO^T into
//   double-buffered TMEM, and accumulating dV += P^T dO and dK += dS^T Q in TMEM with P^T
//   and dS^T written back to TMEM as bf16 (tcgen05.mma with A from TMEM).  The epilogue
//   adds a prompt tile into the fp32 accumulators (read-modify-write by the one CTA that
//   owns the tile: no atomics, stream-ordered across calls) or stores a suffix tile in bf16.
// K4 attn_bwd_dq (query-tile outer): a work unit is one 128-row Q tile; it sweeps 64-key
//   steps over the prompt and the causal suffix, recomputing S and dP and accumulating
//   dQ += dS K in TMEM.  Splitting dQ from dK/dV costs three extra MMAs per tile pair but
//   removes every dQ atomic (the prompt dimension is ~170x the suffix at a 2M prompt).
//
// Both kernels: warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = TMEM owner,
// warps 4-11 = two softmax warpgroups.  Both warpgroups work on every double-buffered TMEM
// tile, each on half of its columns, which halves the softmax latency on the MMA's
// critical path (S/dP of step j -> dS of step j -> the accumulate MMA of step j).
// Every wait is bounded (status word + clean exit on timeout).
#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {
namespace {

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

// =======================================================================================
// K3: dK / dV
// =======================================================================================
template <int D>
struct DkdvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kKV = 128 * D * 2;         // K or V tile, 128 keys
  static constexpr int kSub = 64 * D * 2;         // Q or dO sub-tile, 64 rows
  static constexpr int kNS = 4;                   // sub-tile ring stages
  static constexpr int kStage = 2 * kSub + 1024;  // Q, dO, row stats (512 B, padded)
  static constexpr int kOffK = 0, kOffV = kKV, kOffStage = 2 * kKV;
  static constexpr int kOffBar = kOffStage + kNS * kStage;
  static constexpr int kBarKVFull = 0, kBarKVEmpty = 1, kBarQFull = 2;
  static constexpr int kBarQEmpty = kBarQFull + kNS;
  static constexpr int kBarSFull = kBarQEmpty + kNS;
  static constexpr int kBarDSFull = kBarSFull + 2;
  static constexpr int kBarAccDone = kBarDSFull + 2;
  static constexpr int kBarAccFree = kBarAccDone + 1;
  static constexpr int kBarDrain = kBarAccFree + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
  // TMEM: S^T_b at 64 b, dP^T_b at 128 + 64 b, dV at 256, dK at 256 + D.  Packed bf16
  // P^T / dS^T of rows [32 w, 32 w + 32) alias columns [32 w, 32 w + 16) of S^T_b / dP^T_b.
  __host__ __device__ static constexpr uint32_t col_s(int b) { return 64u * b; }
  __host__ __device__ static constexpr uint32_t col_dp(int b) { return 128u + 64u * b; }
  static constexpr uint32_t kColDV = 256u;
  static constexpr uint32_t kColDK = 256u + D;
};

struct KvUnit {
  int kv;
  bool prompt;
  int key0;   // first key of the tile (prompt or suffix index)
  int i0;     // first 64-row sub-tile
  int n;      // number of sub-tiles
};

__device__ __forceinline__ KvUnit make_kv_unit(int u, const AttnShape& sh, int qt64, int n_q64) {
  const int n_pt = static_cast<int>((sh.P + 127) / 128);
  const int n_st = static_cast<int>((sh.R + 127) / 128);
  KvUnit w;
  w.kv = u / (n_pt + n_st);
  const int j = u - w.kv * (n_pt + n_st);
  w.prompt = j < n_pt;
  w.key0 = w.prompt ? 128 * j : 128 * (j - n_pt);
  w.i0 = w.prompt ? 0 : w.key0 / qt64;
  w.n = n_q64 - w.i0;
  return w;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_kp,
                         const __grid_constant__ CUtensorMap tm_vp,
                         const __grid_constant__ CUtensorMap tm_ks,
                         const __grid_constant__ CUtensorMap tm_vs,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do, const AttnShape sh,
                         const int qt64, const float2* __restrict__ rowstats,
                         float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                         uint16_t* __restrict__ dk_suf, uint16_t* __restrict__ dv_suf,
                         uint32_t* status) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_q64 = static_cast<int>((sh.R + qt64 - 1) / qt64);
  const int n_units =
      sh.Hkv * static_cast<int>((sh.P + 127) / 128 + (sh.R + 127) / 128);
  const int rows_used = sh.g * qt64;   // rows of a 64-row sub-tile that TMA fills

  // Padding rows of every Q/dO stage are never written by TMA: zero them once so that
  // they contribute exactly nothing to the sums over rows in dK and dV.
  if (rows_used < 64) {
    const int pad_rows = 64 - rows_used;
    const int per_stage = 2 * C::kBoxes * pad_rows * 8;   // 16-byte chunks
    for (int idx = threadIdx.x; idx < C::kNS * per_stage; idx += kThreads) {
      const int st = idx / per_stage;
      int rem = idx - st * per_stage;
      const int buf = rem / (C::kBoxes * pad_rows * 8);   // 0 = Q, 1 = dO
      rem -= buf * (C::kBoxes * pad_rows * 8);
      const int box = rem / (pad_rows * 8);
      rem -= box * (pad_rows * 8);
      const int row = rows_used + rem / 8, chunk = rem & 7;
      uint8_t* p = smem + C::kOffStage + st * C::kStage + buf * C::kSub + box * 8192 +
                   row * 128 + chunk * 16;
      *reinterpret_cast<uint4*>(p) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[C::kBarKVFull], 1);
    mbar_init(&bars[C::kBarKVEmpty], 1);
    for (int i = 0; i < C::kNS; ++i) {
      mbar_init(&bars[C::kBarQFull + i], 1);
      mbar_init(&bars[C::kBarQEmpty + i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[C::kBarSFull + b], 1);
      mbar_init(&bars[C::kBarDSFull + b], 256);
    }
    mbar_init(&bars[C::kBarAccDone], 1);
    mbar_init(&bars[C::kBarAccFree], 256);
    mbar_init(&bars[C::kBarDrain], 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    __syncwarp();
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* vabort = &abort_flag;
  const uint32_t q_tx = static_cast<uint32_t>(2 * C::kBoxes * 128 * rows_used + 512);

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      tma_prefetch_desc(&tm_vp);
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      uint32_t qit = 0, uc = 0;
      bool ok = true, kv_pending = false;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const KvUnit w = make_kv_unit(u, sh, qt64, n_q64);
        if (uc > 0) ok = mbar_wait(&bars[C::kBarKVEmpty], (uc - 1) & 1u, status, vabort);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[C::kBarKVFull], 2 * C::kKV);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(smem + C::kOffK + b * 16384, w.prompt ? &tm_kp : &tm_ks,
                      &bars[C::kBarKVFull], 64 * b, w.kv, w.key0);
          tma_load_3d(smem + C::kOffV + b * 16384, w.prompt ? &tm_vp : &tm_vs,
                      &bars[C::kBarKVFull], 64 * b, w.kv, w.key0);
        }
        kv_pending = true;
        for (int li = 0; li < w.n && ok; ++li, ++qit) {
          const int i = w.i0 + li;
          const uint32_t st = qit % C::kNS;
          if (qit >= static_cast<uint32_t>(C::kNS))
            ok = mbar_wait(&bars[C::kBarQEmpty + st], ((qit / C::kNS) - 1) & 1u, status, vabort);
          if (!ok) break;
          uint8_t* base = smem + C::kOffStage + st * C::kStage;
          mbar_arrive_expect_tx(&bars[C::kBarQFull + st], q_tx);
          for (int b = 0; b < C::kBoxes; ++b) {
            tma_load_3d(base + b * 8192, &tm_q, &bars[C::kBarQFull + st], 64 * b, w.kv * sh.g,
                        i * qt64);
            tma_load_3d(base + C::kSub + b * 8192, &tm_do, &bars[C::kBarQFull + st], 64 * b,
                        w.kv * sh.g, i * qt64);
          }
          bulk_load(base + 2 * C::kSub, rowstats + (static_cast<int64_t>(w.kv) * n_q64 + i) * 64,
                    512, &bars[C::kBarQFull + st]);
        }
      }
      if (!ok) {
        *vabort = 1;
        // drain this thread's own copies still in flight (the last kNS issues)
        for (uint32_t it = qit > static_cast<uint32_t>(C::kNS) ? qit - C::kNS : 0u; it < qit; ++it)
          mbar_wait_ns(&bars[C::kBarQFull + it % C::kNS], (it / C::kNS) & 1u, 200000000ull);
        if (kv_pending) mbar_wait_ns(&bars[C::kBarKVFull], (uc) & 1u, 200000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      const uint32_t sStage = smem_u32(smem + C::kOffStage);
      uint32_t qit = 0, uc = 0, dsph = 0u;   // bit b: parity of the next wait on buffer b
      bool ok = true;
      const uint64_t dK0 = smem_desc(sK, 16, 1024), dV0 = smem_desc(sV, 16, 1024);
      const uint64_t dS0 = smem_desc(sStage, 16, 1024);         // K-major view of a stage
      const uint64_t dM0 = smem_desc(sStage, 8192, 1024);       // MN-major view of a stage
      auto issue_s = [&](int b, uint32_t st) {
        const uint64_t q = dS0 + static_cast<uint64_t>((st * C::kStage) >> 4);
        const uint64_t o = q + static_cast<uint64_t>(C::kSub >> 4);
        const uint32_t ds = tmem + C::col_s(b), dp = tmem + C::col_dp(b);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
          mma_bf16_ss(ds, dK0 + oa, q + ob, kIdS, kk > 0 ? 1u : 0u);
          mma_bf16_ss(dp, dV0 + oa, o + ob, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_acc = [&](int b, uint32_t st, bool acc) {
        const uint64_t q = dM0 + static_cast<uint64_t>((st * C::kStage) >> 4);
        const uint64_t o = q + static_cast<uint64_t>(C::kSub >> 4);
        const uint32_t ps = tmem + C::col_s(b), pd = tmem + C::col_dp(b);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // rows 16 kk .. 16 kk + 15: packed by warpgroup kk / 2 at column 32 (kk / 2)
          const uint32_t ac = 32u * (kk >> 1) + 8u * (kk & 1);
          const uint64_t ok_ = static_cast<uint64_t>((kk * 2048) >> 4);
          mma_bf16_ts(tmem + C::kColDV, ps + ac, o + ok_, kIdAcc, (acc || kk > 0) ? 1u : 0u);
          mma_bf16_ts(tmem + C::kColDK, pd + ac, q + ok_, kIdAcc, (acc || kk > 0) ? 1u : 0u);
        }
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const KvUnit w = make_kv_unit(u, sh, qt64, n_q64);
        ok = mbar_wait(&bars[C::kBarKVFull], uc & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        const int npro = w.n < 2 ? w.n : 2;
        for (int b = 0; b < npro && ok; ++b) {
          const uint32_t st = (qit + b) % C::kNS;
          ok = mbar_wait(&bars[C::kBarQFull + st], ((qit + b) / C::kNS) & 1u, status, vabort);
          if (!ok) break;
          tc_fence_after();
          issue_s(b, st);
          mma_commit(&bars[C::kBarSFull + b]);
        }
        for (int li = 0; li < w.n && ok; ++li) {
          const int b = li & 1;
          const uint32_t st = (qit + li) % C::kNS;
          ok = mbar_wait(&bars[C::kBarDSFull + b], (dsph >> b) & 1u, status, vabort);
          if (!ok) break;
          dsph ^= 1u << b;
          if (li == 0 && uc > 0) {
            ok = mbar_wait(&bars[C::kBarAccFree], (uc - 1) & 1u, status, vabort);
            if (!ok) break;
          }
          tc_fence_after();
          issue_acc(b, st, li > 0);
          mma_commit(&bars[C::kBarQEmpty + st]);
          if (li + 2 < w.n) {
            const uint32_t st2 = (qit + li + 2) % C::kNS;
            ok = mbar_wait(&bars[C::kBarQFull + st2], ((qit + li + 2) / C::kNS) & 1u, status,
                           vabort);
            if (!ok) break;
            tc_fence_after();
            issue_s(b, st2);
            mma_commit(&bars[C::kBarSFull + b]);
          }
        }
        if (!ok) break;
        qit += w.n;
        mma_commit(&bars[C::kBarAccDone]);
        if (u + static_cast<int>(gridDim.x) < n_units) mma_commit(&bars[C::kBarKVEmpty]);
      }
      if (!ok) *vabort = 1;
      mma_commit(&bars[C::kBarDrain]);
      mbar_wait_ns(&bars[C::kBarDrain], 0u, ok ? LS_WAIT_LIMIT_NS : 200000000ull);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // key within the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = sh.scale * kLog2e;
    uint32_t sph = 0u, qit = 0u, uc = 0u;   // bit b: parity of the next wait on buffer b
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const KvUnit w = make_kv_unit(u, sh, qt64, n_q64);
      const int key = w.key0 + row;
      // both warpgroups work on every sub-tile: warpgroup wg owns its rows [32 wg, 32 wg + 32)
      for (int li = 0; li < w.n; ++li) {
        const int b = li & 1;
        const uint32_t st = (qit + li) % C::kNS;
        ok = mbar_wait(&bars[C::kBarSFull + b], (sph >> b) & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        sph ^= 1u << b;
        // acquire the row stats copied into this stage (long complete: the MMA waited on it)
        ok = mbar_wait(&bars[C::kBarQFull + st], ((qit + li) / C::kNS) & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float4* rs4 = reinterpret_cast<const float4*>(smem + C::kOffStage + st * C::kStage +
                                                            2 * C::kSub);
        // causal suffix: rows r < lo see only suffix keys < this key
        int lo = 0;
        if (!w.prompt) {
          const int v = sh.g * (key - (w.i0 + li) * qt64);
          lo = v < 0 ? 0 : (v > 64 ? 64 : v);
        }
        uint32_t sv[32], dv[32];
        tmem_ld32(lane_base + C::col_s(b) + wg * 32, sv);
        tmem_ld32(lane_base + C::col_dp(b) + wg * 32, dv);
        tmem_ld_wait();
        float p[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 st4 = rs4[wg * 16 + i];   // (LSE2, Delta) of rows c and c + 1
          p[2 * i] = ex2_approx(fmaf(__uint_as_float(sv[2 * i]), c2, -st4.x));
          p[2 * i + 1] = ex2_approx(fmaf(__uint_as_float(sv[2 * i + 1]), c2, -st4.z));
          dv[2 * i] = __float_as_uint(__uint_as_float(dv[2 * i]) - st4.y);
          dv[2 * i + 1] = __float_as_uint(__uint_as_float(dv[2 * i + 1]) - st4.w);
        }
        if (lo > wg * 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (wg * 32 + i < lo) p[i] = 0.0f;
        }
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pw[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
          dw[i] = pack_bf16x2(p[2 * i] * __uint_as_float(dv[2 * i]),
                              p[2 * i + 1] * __uint_as_float(dv[2 * i + 1]));
        }
        // packed P^T / dS^T go to the first 16 of this warpgroup's own 32 columns, so no
        // write can land on fp32 columns the other warpgroup has yet to read
        tmem_st16(lane_base + C::col_s(b) + wg * 32, pw);
        tmem_st16(lane_base + C::col_dp(b) + wg * 32, dw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[C::kBarDSFull + b]);
      }
      if (!ok) break;
      qit += w.n;
      // epilogue: warpgroup 0 owns dV, warpgroup 1 owns dK
      ok = mbar_wait(&bars[C::kBarAccDone], uc & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool valid = w.prompt ? (key < sh.P) : (key < sh.R);
      const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
      const float mul = wg == 0 ? 1.0f : sh.scale;
      const int64_t off = (static_cast<int64_t>(key) * sh.Hkv + w.kv) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(lane_base + col + cc * 32, v);
        tmem_ld_wait();
        if (valid) {
          if (w.prompt) {
            float4* dst = reinterpret_cast<float4*>((wg == 0 ? dv_acc : dk_acc) + off + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float4 a = dst[i];
              a.x = fmaf(__uint_as_float(v[4 * i + 0]), mul, a.x);
              a.y = fmaf(__uint_as_float(v[4 * i + 1]), mul, a.y);
              a.z = fmaf(__uint_as_float(v[4 * i + 2]), mul, a.z);
              a.w = fmaf(__uint_as_float(v[4 * i + 3]), mul, a.w);
              dst[i] = a;
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>((wg == 0 ? dv_suf : dk_suf) + off + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(v[8 * i + 0]) * mul, __uint_as_float(v[8 * i + 1]) * mul);
              pk.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * mul, __uint_as_float(v[8 * i + 3]) * mul);
              pk.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * mul, __uint_as_float(v[8 * i + 5]) * mul);
              pk.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * mul, __uint_as_float(v[8 * i + 7]) * mul);
              dst[i] = pk;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[C::kBarAccFree]);
    }
    if (!ok) *vabort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =======================================================================================
// K4: dQ
// =======================================================================================
template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kQ = 128 * D * 2;           // Q or dO tile, 128 rows
  static constexpr int kKV = 64 * D * 2;           // K or V step tile, 64 keys
  static constexpr int kNS = (D == 128) ? 4 : 8;   // K/V ring stages
  static constexpr int kStage = 2 * kKV;
  static constexpr int kOffQ = 0, kOffDO = kQ, kOffStage = 2 * kQ;
  static constexpr int kOffBar = kOffStage + kNS * kStage;
  static constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarQTmem = 2, kBarKVFull = 3;
  static constexpr int kBarKVEmpty = kBarKVFull + kNS;
  static constexpr int kBarSFull = kBarKVEmpty + kNS;
  static constexpr int kBarDSFull = kBarSFull + 2;
  static constexpr int kBarDQDone = kBarDSFull + 2;
  static constexpr int kBarDQFree = kBarDQDone + 1;
  static constexpr int kBarDrain = kBarDQFree + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
  // TMEM: S_b at 64 b (packed dS of keys [32 w, 32 w + 32) aliases its columns
  // [32 w, 32 w + 16)), dP_b at 128 + 64 b, dQ at 256,
  // and the unit's Q and dO rows (bf16, the A operand of S = Q K^T and dP = dO V^T) at
  // 384 and 384 + D/2, so those MMAs read only the 64-key K/V tile from shared memory.
  __host__ __device__ static constexpr uint32_t col_s(int b) { return 64u * b; }
  __host__ __device__ static constexpr uint32_t col_dp(int b) { return 128u + 64u * b; }
  static constexpr uint32_t kColDQ = 256u;
  static constexpr uint32_t kColQ = 384u;
  static constexpr uint32_t kColDO = 384u + D / 2;
};

struct QUnit {
  int kv;
  int t0;      // first query of the tile
  int n_pt;    // prompt 64-key steps
  int n;       // total steps
};

__device__ __forceinline__ QUnit make_q_unit(int u, const AttnShape& sh, int n_qt) {
  QUnit w;
  w.kv = u / n_qt;
  const int i = u - w.kv * n_qt;
  w.t0 = i * sh.qt;
  int t_end = w.t0 + sh.qt;
  if (t_end > sh.R) t_end = static_cast<int>(sh.R);
  w.n_pt = static_cast<int>((sh.P + 63) / 64);
  w.n = w.n_pt + (t_end + 63) / 64;
  return w;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_kp,
                       const __grid_constant__ CUtensorMap tm_vp,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do, const AttnShape sh,
                       const int qt64, const float2* __restrict__ rowstats,
                       uint16_t* __restrict__ dq, uint32_t* status) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = static_cast<int>((sh.R + sh.qt - 1) / sh.qt);
  const int n_q64 = static_cast<int>((sh.R + qt64 - 1) / qt64);
  const int n_units = sh.Hkv * n_qt;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[C::kBarQFull], 1);
    mbar_init(&bars[C::kBarQEmpty], 256);
    mbar_init(&bars[C::kBarQTmem], 256);
    for (int i = 0; i < C::kNS; ++i) {
      mbar_init(&bars[C::kBarKVFull + i], 1);
      mbar_init(&bars[C::kBarKVEmpty + i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[C::kBarSFull + b], 1);
      mbar_init(&bars[C::kBarDSFull + b], 256);
    }
    mbar_init(&bars[C::kBarDQDone], 1);
    mbar_init(&bars[C::kBarDQFree], 256);
    mbar_init(&bars[C::kBarDrain], 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    __syncwarp();
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* vabort = &abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      tma_prefetch_desc(&tm_vp);
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      uint32_t kit = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const QUnit w = make_q_unit(u, sh, n_qt);
        if (uc > 0) ok = mbar_wait(&bars[C::kBarQEmpty], (uc - 1) & 1u, status, vabort);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[C::kBarQFull],
                              static_cast<uint32_t>(2 * C::kBoxes * 128 * sh.g * sh.qt));
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(smem + C::kOffQ + b * 16384, &tm_q, &bars[C::kBarQFull], 64 * b,
                      w.kv * sh.g, w.t0);
          tma_load_3d(smem + C::kOffDO + b * 16384, &tm_do, &bars[C::kBarQFull], 64 * b,
                      w.kv * sh.g, w.t0);
        }
        for (int j = 0; j < w.n && ok; ++j, ++kit) {
          const uint32_t st = kit % C::kNS;
          if (kit >= static_cast<uint32_t>(C::kNS))
            ok = mbar_wait(&bars[C::kBarKVEmpty + st], ((kit / C::kNS) - 1) & 1u, status, vabort);
          if (!ok) break;
          const bool pre = j < w.n_pt;
          const int key0 = pre ? 64 * j : 64 * (j - w.n_pt);
          uint8_t* base = smem + C::kOffStage + st * C::kStage;
          mbar_arrive_expect_tx(&bars[C::kBarKVFull + st], 2 * C::kKV);
          for (int b = 0; b < C::kBoxes; ++b) {
            tma_load_3d(base + b * 8192, pre ? &tm_kp : &tm_ks, &bars[C::kBarKVFull + st], 64 * b,
                        w.kv, key0);
            tma_load_3d(base + C::kKV + b * 8192, pre ? &tm_vp : &tm_vs,
                        &bars[C::kBarKVFull + st], 64 * b, w.kv, key0);
          }
        }
      }
      if (!ok) {
        *vabort = 1;
        for (uint32_t it = kit > static_cast<uint32_t>(C::kNS) ? kit - C::kNS : 0u; it < kit; ++it)
          mbar_wait_ns(&bars[C::kBarKVFull + it % C::kNS], (it / C::kNS) & 1u, 200000000ull);
        mbar_wait_ns(&bars[C::kBarQFull], (uc) & 1u, 200000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);
      const uint32_t sStage = smem_u32(smem + C::kOffStage);
      const uint64_t dK0 = smem_desc(sStage, 16, 1024);     // K-major view of a stage
      const uint64_t dM0 = smem_desc(sStage, 8192, 1024);   // MN-major view of a stage
      uint32_t kit = 0, uc = 0, dsph = 0u;   // bit b: parity of the next wait on buffer b
      bool ok = true;
      auto issue_s = [&](int b, uint32_t st) {
        const uint64_t k = dK0 + static_cast<uint64_t>((st * C::kStage) >> 4);
        const uint64_t v = k + static_cast<uint64_t>(C::kKV >> 4);
        const uint32_t ds = tmem + C::col_s(b), dp = tmem + C::col_dp(b);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
          mma_bf16_ts(ds, tmem + C::kColQ + kk * 8, k + ob, kIdS, kk > 0 ? 1u : 0u);
          mma_bf16_ts(dp, tmem + C::kColDO + kk * 8, v + ob, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dq = [&](int b, uint32_t st, bool acc) {
        const uint64_t k = dM0 + static_cast<uint64_t>((st * C::kStage) >> 4);
        const uint32_t a = tmem + C::col_s(b);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // keys 16 kk ..: packed by warpgroup kk / 2 at column 32 (kk / 2)
          mma_bf16_ts(tmem + C::kColDQ, a + 32u * (kk >> 1) + 8u * (kk & 1),
                      k + static_cast<uint64_t>((kk * 2048) >> 4), kIdQ, (acc || kk > 0) ? 1u : 0u);
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const QUnit w = make_q_unit(u, sh, n_qt);
        ok = mbar_wait(&bars[C::kBarQTmem], uc & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        const int npro = w.n < 2 ? w.n : 2;
        for (int b = 0; b < npro && ok; ++b) {
          const uint32_t st = (kit + b) % C::kNS;
          ok = mbar_wait(&bars[C::kBarKVFull + st], ((kit + b) / C::kNS) & 1u, status, vabort);
          if (!ok) break;
          tc_fence_after();
          issue_s(b, st);
          mma_commit(&bars[C::kBarSFull + b]);
        }
        for (int j = 0; j < w.n && ok; ++j) {
          const int b = j & 1;
          const uint32_t st = (kit + j) % C::kNS;
          ok = mbar_wait(&bars[C::kBarDSFull + b], (dsph >> b) & 1u, status, vabort);
          if (!ok) break;
          dsph ^= 1u << b;
          if (j == 0 && uc > 0) {
            ok = mbar_wait(&bars[C::kBarDQFree], (uc - 1) & 1u, status, vabort);
            if (!ok) break;
          }
          tc_fence_after();
          issue_dq(b, st, j > 0);
          mma_commit(&bars[C::kBarKVEmpty + st]);
          if (j + 2 < w.n) {
            const uint32_t st2 = (kit + j + 2) % C::kNS;
            ok = mbar_wait(&bars[C::kBarKVFull + st2], ((kit + j + 2) / C::kNS) & 1u, status,
                           vabort);
            if (!ok) break;
            tc_fence_after();
            issue_s(b, st2);
            mma_commit(&bars[C::kBarSFull + b]);
          }
        }
        if (!ok) break;
        kit += w.n;
        mma_commit(&bars[C::kBarDQDone]);
      }
      if (!ok) *vabort = 1;
      mma_commit(&bars[C::kBarDrain]);
      mbar_wait_ns(&bars[C::kBarDrain], 0u, ok ? LS_WAIT_LIMIT_NS : 200000000ull);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = sh.scale * kLog2e;
    uint32_t sph = 0u, uc = 0u;   // bit b: parity of the next wait on buffer b
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const QUnit w = make_q_unit(u, sh, n_qt);
      const int t = w.t0 + row / sh.g;
      const int hg = row % sh.g;
      const bool valid = (row < sh.g * sh.qt) && (t < sh.R);
      float2 st2 = make_float2(INFINITY, 0.0f);
      if (valid) {
        const int i64 = t / qt64;
        const int r64 = (t - i64 * qt64) * sh.g + hg;
        st2 = rowstats[(static_cast<int64_t>(w.kv) * n_q64 + i64) * 64 + r64];
      }
      // stage this unit's Q (warpgroup 0) or dO (warpgroup 1) row into TMEM; the previous
      // unit's MMAs have all completed (its dQ-done barrier was waited on)
      ok = mbar_wait(&bars[C::kBarQFull], uc & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      {
        const uint8_t* src = smem + (wg == 0 ? C::kOffQ : C::kOffDO);
        const uint32_t col = wg == 0 ? C::kColQ : C::kColDO;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          uint32_t v32[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + bx * 16384 + sw128_offset(row, c));
            v32[4 * c + 0] = v.x;
            v32[4 * c + 1] = v.y;
            v32[4 * c + 2] = v.z;
            v32[4 * c + 3] = v.w;
          }
          tmem_st32(lane_base + col + bx * 32, v32);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[C::kBarQTmem]);
        mbar_arrive(&bars[C::kBarQEmpty]);
      }
      // both warpgroups work on every step: warpgroup wg owns key columns [32 wg, 32 wg + 32)
      for (int j = 0; j < w.n; ++j) {
        const int b = j & 1;
        ok = mbar_wait(&bars[C::kBarSFull + b], (sph >> b) & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        sph ^= 1u << b;
        tc_fence_after();
        int lim = 64;
        if (j < w.n_pt) {
          const int64_t rem = sh.P - 64ll * j;
          if (rem < 64) lim = static_cast<int>(rem);
        } else {
          const int v = t - 64 * (j - w.n_pt) + 1;
          lim = v < 0 ? 0 : (v > 64 ? 64 : v);
        }
        uint32_t sv[32], dv[32];
        tmem_ld32(lane_base + C::col_s(b) + wg * 32, sv);
        tmem_ld32(lane_base + C::col_dp(b) + wg * 32, dv);
        tmem_ld_wait();
        float p[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          p[i] = ex2_approx(fmaf(__uint_as_float(sv[i]), c2, -st2.x));
        if (lim < wg * 32 + 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (wg * 32 + i >= lim) p[i] = 0.0f;
        }
        uint32_t dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          dw[i] = pack_bf16x2(p[2 * i] * (__uint_as_float(dv[2 * i]) - st2.y),
                              p[2 * i + 1] * (__uint_as_float(dv[2 * i + 1]) - st2.y));
        // packed dS goes to the first 16 of this warpgroup's own 32 columns (no write lands
        // on fp32 columns the other warpgroup has yet to read)
        tmem_st16(lane_base + C::col_s(b) + wg * 32, dw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[C::kBarDSFull + b]);
      }
      if (!ok) break;
      // epilogue: dQ * s -> bf16; warpgroup 0 stores columns [0, D/2), warpgroup 1 the rest
      ok = mbar_wait(&bars[C::kBarDQDone], uc & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int h = w.kv * sh.g + hg;
      uint16_t* drow = dq + (static_cast<int64_t>(t) * sh.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = wg * (D / 2) + cc * 32;
        uint32_t v[32];
        tmem_ld32(lane_base + C::kColDQ + col, v);
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(drow + col);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(v[8 * i + 0]) * sh.scale, __uint_as_float(v[8 * i + 1]) * sh.scale);
            pk.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * sh.scale, __uint_as_float(v[8 * i + 3]) * sh.scale);
            pk.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * sh.scale, __uint_as_float(v[8 * i + 5]) * sh.scale);
            pk.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * sh.scale, __uint_as_float(v[8 * i + 7]) * sh.scale);
            dst[i] = pk;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[C::kBarDQFree]);
    }
    if (!ok) *vabort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& a, cudaStream_t s) {
  using C = DkdvCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t n_units = static_cast<int64_t>(a.sh.Hkv) * ((a.sh.P + 127) / 128 + (a.sh.R + 127) / 128);
  int grid = num_sms();
  if (n_units < grid) grid = static_cast<int>(n_units);
  attn_bwd_dkdv_kernel<D><<<grid, kThreads, C::kSmem, s>>>(
      *a.tm_kp128, *a.tm_vp128, a.tm_ks128, a.tm_vs128, a.tm_q64, a.tm_do64, a.sh, a.qt64,
      a.rowstats, a.dk_acc, a.dv_acc, a.dk_suf, a.dv_suf, a.status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_d(const BwdArgs& a, cudaStream_t s) {
  using C = DqCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t n_units = static_cast<int64_t>(a.sh.Hkv) * ((a.sh.R + a.sh.qt - 1) / a.sh.qt);
  int grid = num_sms();
  if (n_units < grid) grid = static_cast<int>(n_units);
  attn_bwd_dq_kernel<D><<<grid, kThreads, C::kSmem, s>>>(*a.tm_kp64, *a.tm_vp64, a.tm_ks64,
                                                        a.tm_vs64, a.tm_q128, a.tm_do128, a.sh,
                                                        a.qt64, a.rowstats, a.dq, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  return a.sh.D == 128 ? launch_dkdv_d<128>(a, s) : launch_dkdv_d<64>(a, s);
}

cudaError_t launch_attn_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  return a.sh.D == 128 ? launch_dq_d<128>(a, s) : launch_dq_d<64>(a, s);
}

}  // namespace ls
