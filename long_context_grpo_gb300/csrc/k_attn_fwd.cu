// K1: forward replay of one response against the resident prompt (LongStraw review,
// dimensionstp.github.io "LongStraw", section 2-1 step 4 "serial policy replay" and
// section 3-2 (4)): for every suffix row t and query head h,
//   O[t,h] = softmax(s q_{t,h} . [K_prompt ; K_suffix[0..t]]) [V_prompt ; V_suffix[0..t]]
//   LSE[t,h] = log sum exp(s q . k).
//
// GB300 design (one persistent CTA per SM, 384 threads):
//   warp 0        TMA producer: two Q tiles per work unit, then K and V tiles (128 keys)
//                 into separate 2-stage rings (prompt keys first, then the causal suffix).
//   warp 1        issues tcgen05.mma as a converged warp (one elected lane issues, every
//                 lane polls the waits): S_q = Q_q K^T into TMEM (fp32, 128 cols) and
//                 O_q += P_q V with P_q read back from TMEM (bf16, aliasing S_q), each
//                 64-key half of P_q as soon as the softmax has signalled it.
//   warp 2        allocates / frees the 512 TMEM columns.
//   warps 4-7,    softmax warpgroups, one per Q tile; thread = TMEM lane = tile row.
//   warps 8-11    Online softmax in log2 units with a lazy rescale: the running max only
//                 moves when a tile's max exceeds it by more than 2^8, and only then is
//                 the O row in TMEM rescaled.
// A work unit is (kv head, pair of 128-row Q tiles); each 128-row tile packs qt = 128/g
// consecutive queries x the g query heads that share the kv head, so one K/V tile feeds
// 2 x 128 rows of MMA.  Units are ordered kv-head-major so the CTAs running at the same
// time stream the same prompt K/V through L2.
// Instantiations: <D, kPacked, kNoSuffix>.  kPacked: several responses packed along the
// token axis (units, Q rows and suffix keys offset by the response's packed row; each
// response sees the prompt and only its own causal suffix).  kNoSuffix: prompt keys only
// (one shard of a context-parallel prompt).  <D, false, false> is the one-response replay.
// Every wait is bounded; on a timeout the CTA records it in the status word, drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {
namespace {

constexpr int kThreads = 384;
// Suspend-time hints (ns) of each role's mbarrier waits (0: the hardware's own limit).
// A 20 ns hint on every role measured 3.6 % faster than none for this kernel at a 2M prompt
// (A/B on one GB300); per-role hints alone did not help, and the backward kernels are
// faster without (their constants stay 0).
constexpr uint32_t kHintFwdProducer = 20u, kHintFwdMma = 20u, kHintFwdSoftmax = 20u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;          // bytes of a 128-row bf16 tile
  static constexpr int kNK = (D == 128) ? 2 : 4;     // K ring stages
  static constexpr int kNV = (D == 128) ? 2 : 4;     // V ring stages
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kNK * kTile;
  static constexpr int kOffBar = kOffV + kNV * kTile;
  // barriers: q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
  //           s_full[2], p_full[2][2] (per tile, per 64-key half), o_done[2], o_free[2],
  //           drain
  static constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarKFull = 2;
  static constexpr int kBarKEmpty = kBarKFull + kNK;
  static constexpr int kBarVFull = kBarKEmpty + kNK;
  static constexpr int kBarVEmpty = kBarVFull + kNV;
  static constexpr int kBarSFull = kBarVEmpty + kNV;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarODone = kBarPFull + 4;
  static constexpr int kBarOFree = kBarODone + 2;
  static constexpr int kBarDrain = kBarOFree + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
  // TMEM columns: S_q at 128 q (P_q aliases its first 64 columns), O_q at 256 + D q
  __host__ __device__ static constexpr uint32_t col_s(int q) { return 128u * q; }
  __host__ __device__ static constexpr uint32_t col_o(int q) { return 256u + D * q; }
};

struct Unit {
  int kv;
  int base;      // packed row of the response's first token
  int R;         // response length
  int t0;        // first query of Q tile 0 (response-local)
  bool has1;     // Q tile 1 exists
  int n_pt;      // prompt key tiles
  int n_kt;      // total key tiles
};

// Flat unit u -> (kv head, pair of Q tiles) of one response (base 0, length sh.R); kv-major
// so concurrently running CTAs stream the same prompt K/V.
__device__ __forceinline__ Unit make_unit(int u, const AttnShape& sh, int n_pairs) {
  Unit w;
  w.kv = u / n_pairs;
  const int pair = u - w.kv * n_pairs;
  const int n_qt = static_cast<int>((sh.R + sh.qt - 1) / sh.qt);
  w.base = 0;
  w.R = static_cast<int>(sh.R);
  w.t0 = pair * 2 * sh.qt;
  w.has1 = (2 * pair + 1) < n_qt;
  int t_end = w.t0 + (w.has1 ? 2 : 1) * sh.qt;
  if (t_end > sh.R) t_end = static_cast<int>(sh.R);
  w.n_pt = static_cast<int>((sh.P + 127) / 128);
  w.n_kt = w.n_pt + (t_end + 127) / 128;
  return w;
}

// Packed responses: flat unit u -> (kv head, response, pair of that response's Q tiles).
__device__ __forceinline__ Unit make_unit_packed(int u, const AttnShape& sh, const Varlen& vl) {
  Unit w;
  const int n_pairs = vl.pair0[vl.G];
  w.kv = u / n_pairs;
  const int x = u - w.kv * n_pairs;
  const int b = varlen_find(vl.pair0, vl.G, x);
  const int pair = x - vl.pair0[b];
  w.base = vl.row0[b];
  w.R = vl.row0[b + 1] - w.base;
  const int n_qt = (w.R + sh.qt - 1) / sh.qt;
  w.t0 = pair * 2 * sh.qt;
  w.has1 = (2 * pair + 1) < n_qt;
  int t_end = w.t0 + (w.has1 ? 2 : 1) * sh.qt;
  if (t_end > w.R) t_end = w.R;
  w.n_pt = static_cast<int>((sh.P + 127) / 128);
  w.n_kt = w.n_pt + (t_end + 127) / 128;
  return w;
}

// kNoSuffix: the queries see the prompt keys only (one shard of a context-parallel prompt).
template <bool kPacked, bool kNoSuffix>
__device__ __forceinline__ Unit pick_unit(int u, const AttnShape& sh, int n_pairs, const Varlen& vl) {
  if constexpr (kPacked) {
    return make_unit_packed(u, sh, vl);
  } else {
    Unit w = make_unit(u, sh, n_pairs);
    if constexpr (kNoSuffix) w.n_kt = w.n_pt;
    return w;
  }
}

template <int D, bool kPacked, bool kNoSuffix>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_kp,
                    const __grid_constant__ CUtensorMap tm_vp,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_ks,
                    const __grid_constant__ CUtensorMap tm_vs, const AttnShape sh,
                    const __grid_constant__ Varlen vl, uint16_t* __restrict__ o_out,
                    float* __restrict__ lse_out, uint32_t* status) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_pairs = kPacked ? vl.pair0[vl.G]
                              : static_cast<int>(((sh.R + sh.qt - 1) / sh.qt + 1) / 2);
  const int n_units = sh.Hkv * n_pairs;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[C::kBarQFull], 1);
    mbar_init(&bars[C::kBarQEmpty], 1);
    for (int i = 0; i < C::kNK; ++i) {
      mbar_init(&bars[C::kBarKFull + i], 1);
      mbar_init(&bars[C::kBarKEmpty + i], 1);
    }
    for (int i = 0; i < C::kNV; ++i) {
      mbar_init(&bars[C::kBarVFull + i], 1);
      mbar_init(&bars[C::kBarVEmpty + i], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars[C::kBarSFull + q], 1);
      mbar_init(&bars[C::kBarPFull + 2 * q], 128);
      mbar_init(&bars[C::kBarPFull + 2 * q + 1], 128);
      mbar_init(&bars[C::kBarODone + q], 1);
      mbar_init(&bars[C::kBarOFree + q], 128);
    }
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      tma_prefetch_desc(&tm_vp);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
      uint32_t kit = 0, vit = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const Unit w = pick_unit<kPacked, kNoSuffix>(u, sh, n_pairs, vl);
        if (uc > 0) ok = mbar_wait_hint<kHintFwdProducer>(&bars[C::kBarQEmpty], (uc - 1) & 1u, status);
        if (!ok) break;
        const int nq = w.has1 ? 2 : 1;
        mbar_arrive_expect_tx(&bars[C::kBarQFull],
                              static_cast<uint32_t>(nq * C::kBoxes * 128 * sh.g * sh.qt));
        for (int q = 0; q < nq; ++q)
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kOffQ + q * C::kTile + b * 16384, &tm_q, &bars[C::kBarQFull],
                        64 * b, w.kv * sh.g, (kPacked ? w.base : 0) + w.t0 + q * sh.qt);
        for (int j = 0; j < w.n_kt && ok; ++j) {
          const bool pre = j < w.n_pt;
          const int key0 = pre ? 128 * j : (kPacked ? w.base : 0) + 128 * (j - w.n_pt);
          {
            const uint32_t s = kit % C::kNK;
            if (kit >= static_cast<uint32_t>(C::kNK))
              ok = mbar_wait_hint<kHintFwdProducer>(&bars[C::kBarKEmpty + s], ((kit / C::kNK) - 1) & 1u, status);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[C::kBarKFull + s], C::kTile);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(smem + C::kOffK + s * C::kTile + b * 16384, pre ? &tm_kp : &tm_ks,
                          &bars[C::kBarKFull + s], 64 * b, w.kv, key0);
            ++kit;
          }
          {
            const uint32_t s = vit % C::kNV;
            if (vit >= static_cast<uint32_t>(C::kNV))
              ok = mbar_wait_hint<kHintFwdProducer>(&bars[C::kBarVEmpty + s], ((vit / C::kNV) - 1) & 1u, status);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[C::kBarVFull + s], C::kTile);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(smem + C::kOffV + s * C::kTile + b * 16384, pre ? &tm_vp : &tm_vs,
                          &bars[C::kBarVFull + s], 64 * b, w.kv, key0);
            ++vit;
          }
        }
      }
      if (!ok) {
        *vabort = 1;
        // drain this thread's own copies still in flight before the CTA may exit
        for (uint32_t it = kit > static_cast<uint32_t>(C::kNK) ? kit - C::kNK : 0u; it < kit; ++it)
          mbar_wait_ns(&bars[C::kBarKFull + it % C::kNK], (it / C::kNK) & 1u, 200000000ull);
        for (uint32_t it = vit > static_cast<uint32_t>(C::kNV) ? vit - C::kNV : 0u; it < vit; ++it)
          mbar_wait_ns(&bars[C::kBarVFull + it % C::kNV], (it / C::kNV) & 1u, 200000000ull);
        mbar_wait_ns(&bars[C::kBarQFull], (uc) & 1u, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::kOffQ);
      const uint32_t sK = smem_u32(smem + C::kOffK);
      const uint32_t sV = smem_u32(smem + C::kOffV);
      uint32_t kit = 0, vit = 0, uc = 0;
      uint32_t pph = 0u;             // bit q: parity of the next p_full wait of tile q
      uint32_t uq0 = 0u, uq1 = 0u;   // units processed per tile
      bool ok = true;

      // Base descriptors; a tile or k-step offset is added to the start-address field
      // (bits 0-13, address >> 4), which cannot carry out for shared addresses < 256 KB.
      const uint64_t dQ0 = smem_desc(sQ, 16, 1024);
      const uint64_t dK0 = smem_desc(sK, 16, 1024);
      const uint64_t dV0 = smem_desc(sV, 16384, 1024);
      auto issue_s = [&](int q, uint32_t kstage) {
        const uint64_t qa = dQ0 + static_cast<uint64_t>((q * C::kTile) >> 4);
        const uint64_t ka = dK0 + static_cast<uint64_t>((kstage * C::kTile) >> 4);
        const uint32_t d = tmem + C::col_s(q);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(d, qa + off, ka + off, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      // O_q (+)= P_q V over keys 64 h .. 64 h + 63 (k-steps 4 h .. 4 h + 3)
      auto issue_pv = [&](int q, uint32_t vstage, int h, bool acc) {
        const uint64_t va = dV0 + static_cast<uint64_t>((vstage * C::kTile) >> 4);
        const uint32_t d = tmem + C::col_o(q), a = tmem + C::col_s(q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = 4 * h + i;
          mma_bf16_ts_w(d, a + kk * 8, va + static_cast<uint64_t>((kk * 2048) >> 4), kIdPV,
                        (acc || i > 0) ? 1u : 0u);
        }
      };

      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const Unit w = pick_unit<kPacked, kNoSuffix>(u, sh, n_pairs, vl);
        const int nq = w.has1 ? 2 : 1;
        ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarQFull], uc & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        // S_q(0)
        uint32_t ks = kit % C::kNK;
        ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarKFull + ks], (kit / C::kNK) & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        for (int q = 0; q < nq; ++q) {
          issue_s(q, ks);
          mma_commit_w(&bars[C::kBarSFull + q]);
        }
        mma_commit_w(&bars[C::kBarKEmpty + ks]);
        ++kit;
        for (int j = 0; j < w.n_kt && ok; ++j) {
          const uint32_t vs = vit % C::kNV;
          ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarVFull + vs], (vit / C::kNV) & 1u, status, vabort);
          if (!ok) break;
          const bool more = (j + 1) < w.n_kt;
          uint32_t ks_next = kit % C::kNK;
          for (int q = 0; q < nq && ok; ++q) {
            ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarPFull + 2 * q], (pph >> q) & 1u, status, vabort);
            if (!ok) break;
            const uint32_t uqq = q ? uq1 : uq0;
            if (j == 0 && uqq > 0) {
              ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarOFree + q], (uqq - 1) & 1u, status, vabort);
              if (!ok) break;
            }
            tc_fence_after();
            issue_pv(q, vs, 0, j > 0);   // runs while the softmax finishes the second half
            ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarPFull + 2 * q + 1], (pph >> q) & 1u, status, vabort);
            if (!ok) break;
            pph ^= 1u << q;
            tc_fence_after();
            issue_pv(q, vs, 1, true);
            if (!more) mma_commit_w(&bars[C::kBarODone + q]);
            if (more) {
              if (q == 0) {
                ok = mbar_wait_warp<kHintFwdMma>(&bars[C::kBarKFull + ks_next], (kit / C::kNK) & 1u, status, vabort);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(q, ks_next);
              mma_commit_w(&bars[C::kBarSFull + q]);
            }
          }
          if (!ok) break;
          if (more) {
            mma_commit_w(&bars[C::kBarKEmpty + ks_next]);
            ++kit;
          }
          mma_commit_w(&bars[C::kBarVEmpty + vs]);
          ++vit;
        }
        if (!ok) break;
        ++uq0;
        if (nq > 1) ++uq1;
        if (u + static_cast<int>(gridDim.x) < n_units) mma_commit_w(&bars[C::kBarQEmpty]);
      }
      if (!ok) *vabort = 1;
      // drain: every MMA (and the arrivals committed behind it) has landed before exit
      mma_commit_w(&bars[C::kBarDrain]);
      mbar_wait_ns(&bars[C::kBarDrain], 0u, ok ? LS_WAIT_LIMIT_NS : 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warpgroups
    const int q = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t colS = C::col_s(q), colO = C::col_o(q);
    const float c2 = sh.scale * kLog2e;
    uint32_t sph = 0u, uq = 0u;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = pick_unit<kPacked, kNoSuffix>(u, sh, n_pairs, vl);
      if (q == 1 && !w.has1) continue;
      const int t = w.t0 + q * sh.qt + row / sh.g;
      float m_run = -INFINITY, l = 0.0f;
      for (int j = 0; j < w.n_kt; ++j) {
        ok = mbar_wait_hint<kHintFwdSoftmax>(&bars[C::kBarSFull + q], sph, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        sph ^= 1u;
        tc_fence_after();
        uint32_t sv[4][32];
        tmem_ld32(lane_base + colS + 0, sv[0]);
        tmem_ld32(lane_base + colS + 32, sv[1]);
        tmem_ld32(lane_base + colS + 64, sv[2]);
        tmem_ld32(lane_base + colS + 96, sv[3]);
        tmem_ld_wait();
        // valid key columns of this row in this tile
        int lim = 128;
        if (j < w.n_pt) {
          const int64_t rem = sh.P - 128ll * j;
          if (rem < 128) lim = static_cast<int>(rem);
        } else {
          const int k0 = 128 * (j - w.n_pt);
          const int v = t - k0 + 1;
          lim = v < 0 ? 0 : (v > 128 ? 128 : v);
        }
        if (lim < 128) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
        }
        // row maximum: four independent chains of three-input maxima (exact in any order),
        // so the dependent chain is 16 deep instead of 64
        float mxa = -INFINITY, mxb = -INFINITY, mxc = -INFINITY, mxd = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mxa = fmax3(mxa, __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c + 1) & 31]));
          mxb = fmax3(mxb, __uint_as_float(sv[c >> 5][(c + 2) & 31]), __uint_as_float(sv[c >> 5][(c + 3) & 31]));
          mxc = fmax3(mxc, __uint_as_float(sv[c >> 5][(c + 4) & 31]), __uint_as_float(sv[c >> 5][(c + 5) & 31]));
          mxd = fmax3(mxd, __uint_as_float(sv[c >> 5][(c + 6) & 31]), __uint_as_float(sv[c >> 5][(c + 7) & 31]));
        }
        const float mx = fmax3(mxa, mxb, fmaxf(mxc, mxd));
        const float mt = mx * c2;
        float factor = 1.0f;
        bool resc = false;
        if (m_run == -INFINITY) {
          m_run = mt;
        } else if (mt > m_run + kRescaleLog2) {
          factor = ex2_approx(m_run - mt);
          l *= factor;
          m_run = mt;
          resc = true;
        }
        const float neg_m = (m_run == -INFINITY) ? 0.0f : -m_run;
        // exponent arguments and the row sum on fp32 pairs (one instruction per two keys);
        // the sum runs in four independent pair accumulators (16-deep dependent chains).
        // Each 64-key half of P is signalled as soon as it is in TMEM, unless a row of this
        // warp raised its running maximum: O is rescaled first then (the P V of this step
        // accumulates into it), and both halves are signalled after that.
        const bool any_resc = __any_sync(0xffffffffu, resc);
        const uint64_t c2x2 = f2_pack(c2, c2), nm2 = f2_pack(neg_m, neg_m);
        uint64_t rs2[4] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f),
                           f2_pack(0.0f, 0.0f)};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pw[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = half * 64 + 2 * i;
            const uint64_t a = f2_fma(f2_pack(__uint_as_float(sv[c >> 5][c & 31]),
                                              __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31])),
                                      c2x2, nm2);
            float x0, x1;
            f2_unpack(a, x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            rs2[i & 3] = f2_add(rs2[i & 3], f2_pack(p0, p1));
            pw[i] = pack_bf16x2(p0, p1);
          }
          tmem_st32(lane_base + colS + half * 32, pw);
          if (!any_resc) {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[C::kBarPFull + 2 * q + half]);
          }
        }
        float rs0, rs1, rs2f, rs3;
        f2_unpack(f2_add(rs2[0], rs2[1]), rs0, rs1);
        f2_unpack(f2_add(rs2[2], rs2[3]), rs2f, rs3);
        l += (rs0 + rs1) + (rs2f + rs3);
        if (any_resc) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(lane_base + colO + cc * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * factor);
            tmem_st32(lane_base + colO + cc * 32, ov);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::kBarPFull + 2 * q]);
          mbar_arrive(&bars[C::kBarPFull + 2 * q + 1]);
        }
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE
      ok = mbar_wait_hint<kHintFwdSoftmax>(&bars[C::kBarODone + q], uq & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool valid = (row < sh.g * sh.qt) && (kPacked ? t < w.R : t < sh.R);
      const int h = w.kv * sh.g + row % sh.g;
      const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
      const int64_t prow = kPacked ? static_cast<int64_t>(w.base) + t : static_cast<int64_t>(t);
      uint16_t* orow = o_out + (prow * sh.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld32(lane_base + colO + cc * 32, ov);
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv_l, __uint_as_float(ov[8 * i + 1]) * inv_l);
            pk.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv_l, __uint_as_float(ov[8 * i + 3]) * inv_l);
            pk.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv_l, __uint_as_float(ov[8 * i + 5]) * inv_l);
            pk.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv_l, __uint_as_float(ov[8 * i + 7]) * inv_l);
            dst[i] = pk;
          }
        }
      }
      if (valid) lse_out[prow * sh.Hq + h] = (m_run + __log2f(l)) * kLn2;
      tc_fence_before();
      mbar_arrive(&bars[C::kBarOFree + q]);
      ++uq;
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

template <int D, bool kPacked, bool kNoSuffix = false>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  // the shared-memory opt-in is per device: remember it per device index
  static bool attr_set[kMaxDeviceCache] = {};
  const int dev = cached_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kPacked, kNoSuffix>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t n_units = static_cast<int64_t>(a.sh.Hkv) * a.vl.pair0[a.vl.G];
  int grid = num_sms();
  if (n_units < grid) grid = static_cast<int>(n_units);
  attn_fwd_kernel<D, kPacked, kNoSuffix><<<grid, kThreads, C::kSmem, s>>>(
      *a.tm_kp, *a.tm_vp, a.tm_q, a.tm_ks, a.tm_vs, a.sh, a.vl, a.o, a.lse, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t s) {
  if (a.no_suffix) return a.sh.D == 128 ? launch_fwd_d<128, false, true>(a, s) : launch_fwd_d<64, false, true>(a, s);
  if (a.vl.G > 1) return a.sh.D == 128 ? launch_fwd_d<128, true>(a, s) : launch_fwd_d<64, true>(a, s);
  return a.sh.D == 128 ? launch_fwd_d<128, false>(a, s) : launch_fwd_d<64, false>(a, s);
}

}  // namespace ls
