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
//   a prompt tile or a suffix tile.  It sweeps every 128-row Q/dO tile that sees its keys
//   (qt = 128/g queries x the g heads of the kv head).  Per tile: S^T = K Q^T and
//   dP^T = V dO^T into TMEM, the softmax turns them into bf16 P^T and dS^T, and
//   dV += P^T dO, dK += dS^T Q accumulate in TMEM (tcgen05.mma with A from TMEM).  The
//   epilogue adds a prompt tile into the fp32 accumulators (read-modify-write by the one CTA
//   that owns the tile: no atomics, stream-ordered across calls) or stores a suffix tile
//   (in block replay the suffix tile is added into the accumulators too, at rows P + key).
// K4 attn_bwd_dq (query-tile outer): a work unit is one 128-row Q tile; it sweeps 128-key
//   steps over the prompt and the causal suffix, recomputing S and dP and accumulating
//   dQ += dS K in TMEM.  Splitting dQ from dK/dV costs recomputing S and dP but removes every
//   dQ atomic (the prompt is ~170x the suffix at a 2M prompt).
//
// Every MMA is 128 x 128 (or 128 x D): narrower tcgen05 tiles run well below the tensor
// rate.  TMEM holds one S and one dP tile; the overlap comes from where the softmax puts its
// bf16 results: packed P/dS overwrite the fp32 dP columns the softmax has just read, so the
// S columns are free as soon as S is in registers and the next tile's S = K Q^T (or Q K^T)
// runs on the tensor pipe while the softmax works; the next dP is issued, in order, after
// the MMAs that read P/dS.  P/dS are signalled per 32-column chunk of each warpgroup, so the
// MMAs over the first chunk's k-steps run while the softmax computes the second.
//
// Warp roles (384 threads, one CTA per SM): warp 0 TMA producer, warp 1 the MMA issuer (a
// converged warp: every lane polls the waits, one elected lane issues each MMA and commit),
// warp 2 TMEM owner, warps 4-11 two softmax warpgroups; warpgroup w owns tile columns
// [64 w, 64 w + 64).  Every wait is bounded (status word + clean exit on timeout).
//
// Instantiations <D, kPacked, kNoSuffix> as in the forward: packed responses (a prompt tile
// then sweeps the Q tiles of every response before its single read-modify-write; Q rows past
// a response's end carry +inf row statistics), or prompt keys only (context-parallel
// shards).
#include "ls_internal.h"
#include "ptx.cuh"

namespace ls {
namespace {

constexpr int kThreads = 384;
// Suspend-time hints (ns) of each role's mbarrier waits (0: the hardware's own limit; a
// 20 ns hint measured slower here, see the forward kernel).
constexpr uint32_t kHintDkdvProducer = 0u, kHintDkdvMma = 0u, kHintDkdvSoftmax = 0u;
constexpr uint32_t kHintDqProducer = 0u, kHintDqMma = 0u, kHintDqSoftmax = 0u;
constexpr float kLog2e = 1.4426950408889634f;

// Column (within a 128-column TMEM region) of the packed bf16 A operand for k-step kk
// (16 rows or keys): warpgroup kk / 4 wrote rows [64 w, 64 w + 64) as two 32-row chunks,
// each chunk's 16 packed columns placed at the start of that chunk's own fp32 columns.
__device__ __forceinline__ constexpr uint32_t packed_col(int kk) {
  return 64u * (kk >> 2) + 32u * ((kk >> 1) & 1) + 8u * (kk & 1);
}

// =======================================================================================
// K3: dK / dV
// =======================================================================================
template <int D>
struct DkdvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = 128 * D * 2;         // K, V, Q or dO tile (128 rows)
  static constexpr int kNQ = 3;                     // Q ring: needed early (S) and late (dK)
  static constexpr int kNO = 2;                     // dO ring: needed by dP and dV
  static constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile;
  static constexpr int kOffO = kOffQ + kNQ * kTile;
  static constexpr int kOffBar = kOffO + kNO * kTile;
  static constexpr int kBarKVFull = 0, kBarKVEmpty = 1, kBarQFull = 2;
  static constexpr int kBarQEmpty = kBarQFull + kNQ;
  static constexpr int kBarOFull = kBarQEmpty + kNQ;
  static constexpr int kBarOEmpty = kBarOFull + kNO;
  static constexpr int kBarSFull = kBarOEmpty + kNO;
  static constexpr int kBarSFree = kBarSFull + 1;
  static constexpr int kBarDPFull = kBarSFree + 1;
  // P/dS written, per 32-column chunk of each warpgroup (chunk c: k-steps with bit 1 = c)
  static constexpr int kBarPDSFull = kBarDPFull + 1;
  static constexpr int kBarAccDone = kBarPDSFull + 2;
  static constexpr int kBarAccFree = kBarAccDone + 1;
  static constexpr int kBarDrain = kBarAccFree + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
  // TMEM: S^T at 0, dP^T at 128 (packed P^T at packed_col(kk), dS^T 16 columns further),
  // dV at 256, dK at 256 + D.
  static constexpr uint32_t kColS = 0u, kColDP = 128u, kColDV = 256u, kColDK = 256u + D;
};

struct KvUnit {
  int kv;
  bool prompt;
  int key0;   // first key of the tile (prompt index, or response-local suffix index)
  int base;   // suffix tiles: packed row of the response's first token
  int R;      // suffix tiles: response length
  int b;      // suffix tiles: response
  int f0;     // first flat 128-row Q tile that sees the tile
  int n;      // number of Q tiles
};

// Flat unit u -> (kv head, 128-key tile).  A prompt tile is seen by every Q tile of every
// packed response; a suffix tile of response b by that response's tiles from the first
// one holding a query at or after its first key.
template <bool kPacked, bool kNoSuffix>
__device__ __forceinline__ KvUnit make_kv_unit(int u, const AttnShape& sh, const Varlen& vl) {
  const int n_pt = static_cast<int>((sh.P + 127) / 128);
  KvUnit w;
  if constexpr (!kPacked) {
    // one response: base 0, length sh.R (kNoSuffix: prompt key tiles only)
    const int n_st = kNoSuffix ? 0 : static_cast<int>((sh.R + 127) / 128);
    const int n_qt = static_cast<int>((sh.R + sh.qt - 1) / sh.qt);
    w.kv = u / (n_pt + n_st);
    const int j = u - w.kv * (n_pt + n_st);
    w.prompt = j < n_pt;
    w.key0 = w.prompt ? 128 * j : 128 * (j - n_pt);
    w.base = 0;
    w.R = static_cast<int>(sh.R);
    w.b = 0;
    w.f0 = w.prompt ? 0 : w.key0 / sh.qt;
    w.n = n_qt - w.f0;
    return w;
  }
  const int n_st = vl.kt0[vl.G];
  w.kv = u / (n_pt + n_st);
  const int j = u - w.kv * (n_pt + n_st);
  w.prompt = j < n_pt;
  if (w.prompt) {
    w.key0 = 128 * j;
    w.base = 0;
    w.R = 0;
    w.b = 0;
    w.f0 = 0;
    w.n = vl.qt0[vl.G];
  } else {
    const int x = j - n_pt;
    w.b = varlen_find(vl.kt0, vl.G, x);
    w.key0 = 128 * (x - vl.kt0[w.b]);
    w.base = vl.row0[w.b];
    w.R = vl.row0[w.b + 1] - w.base;
    w.f0 = vl.qt0[w.b] + w.key0 / sh.qt;
    w.n = vl.qt0[w.b + 1] - w.f0;
  }
  return w;
}

template <int D, bool kPacked, bool kNoSuffix>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_kp,
                         const __grid_constant__ CUtensorMap tm_vp,
                         const __grid_constant__ CUtensorMap tm_ks,
                         const __grid_constant__ CUtensorMap tm_vs,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do, const AttnShape sh,
                         const float* __restrict__ rowstats, float* __restrict__ dk_acc,
                         float* __restrict__ dv_acc, uint16_t* __restrict__ dk_suf,
                         uint16_t* __restrict__ dv_suf, const int suffix_to_acc,
                         const __grid_constant__ Varlen vl, uint32_t* status) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = kPacked ? vl.qt0[vl.G] : static_cast<int>((sh.R + sh.qt - 1) / sh.qt);
  const int n_units = sh.Hkv * (static_cast<int>((sh.P + 127) / 128) +
                                (kPacked ? vl.kt0[vl.G]
                                         : (kNoSuffix ? 0 : static_cast<int>((sh.R + 127) / 128))));
  const int rows_used = sh.g * sh.qt;   // rows of a 128-row tile that TMA fills

  // Padding rows of every Q/dO buffer are never written by TMA: zero them once so that
  // they contribute exactly nothing to the sums over rows in dK and dV.
  if (rows_used < 128) {
    const int pad_rows = 128 - rows_used;
    const int per_buf = C::kBoxes * pad_rows * 8;   // 16-byte chunks per buffer
    for (int idx = threadIdx.x; idx < (C::kNQ + C::kNO) * per_buf; idx += kThreads) {
      const int buf = idx / per_buf;                 // Q ring buffers, then dO ring buffers
      int rem = idx - buf * per_buf;
      const int box = rem / (pad_rows * 8);
      rem -= box * (pad_rows * 8);
      const int row = rows_used + rem / 8, chunk = rem & 7;
      uint8_t* p = smem + C::kOffQ + buf * C::kTile + box * 16384 + row * 128 + chunk * 16;
      *reinterpret_cast<uint4*>(p) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[C::kBarKVFull], 1);
    mbar_init(&bars[C::kBarKVEmpty], 1);
    for (int i = 0; i < C::kNQ; ++i) {
      mbar_init(&bars[C::kBarQFull + i], 1);
      mbar_init(&bars[C::kBarQEmpty + i], 1);
    }
    for (int i = 0; i < C::kNO; ++i) {
      mbar_init(&bars[C::kBarOFull + i], 1);
      mbar_init(&bars[C::kBarOEmpty + i], 1);
    }
    mbar_init(&bars[C::kBarSFull], 1);
    mbar_init(&bars[C::kBarSFree], 256);
    mbar_init(&bars[C::kBarDPFull], 1);
    mbar_init(&bars[C::kBarPDSFull], 256);
    mbar_init(&bars[C::kBarPDSFull + 1], 256);
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
  const uint32_t tile_tx = static_cast<uint32_t>(C::kBoxes * 128 * rows_used);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      tma_prefetch_desc(&tm_vp);
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      uint32_t qit = 0, uc = 0, q_sent = 0;
      bool ok = true, kv_pending = false;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const KvUnit w = make_kv_unit<kPacked, kNoSuffix>(u, sh, vl);
        kv_pending = false;
        if (uc > 0) ok = mbar_wait_hint<kHintDkdvProducer>(&bars[C::kBarKVEmpty], (uc - 1) & 1u, status, vabort);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[C::kBarKVFull], 2 * C::kTile);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(smem + C::kOffK + b * 16384, w.prompt ? &tm_kp : &tm_ks,
                      &bars[C::kBarKVFull], 64 * b, w.kv, w.base + w.key0);
          tma_load_3d(smem + C::kOffV + b * 16384, w.prompt ? &tm_vp : &tm_vs,
                      &bars[C::kBarKVFull], 64 * b, w.kv, w.base + w.key0);
        }
        kv_pending = true;
        int rb = w.prompt ? 0 : w.b;   // response of the current Q tile
        for (int li = 0; li < w.n && ok; ++li, ++qit) {
          const int f = w.f0 + li;
          int qrow = f * sh.qt;         // packed row of the tile
          if constexpr (kPacked) {
            while (f >= vl.qt0[rb + 1]) ++rb;
            qrow = vl.row0[rb] + (f - vl.qt0[rb]) * sh.qt;
          }
          const uint32_t sq = qit % C::kNQ, so = qit % C::kNO;
          if (qit >= static_cast<uint32_t>(C::kNQ))
            ok = mbar_wait_hint<kHintDkdvProducer>(&bars[C::kBarQEmpty + sq], ((qit / C::kNQ) - 1) & 1u, status, vabort);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[C::kBarQFull + sq], tile_tx);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kOffQ + sq * C::kTile + b * 16384, &tm_q,
                        &bars[C::kBarQFull + sq], 64 * b, w.kv * sh.g, qrow);
          ++q_sent;
          if (qit >= static_cast<uint32_t>(C::kNO))
            ok = mbar_wait_hint<kHintDkdvProducer>(&bars[C::kBarOEmpty + so], ((qit / C::kNO) - 1) & 1u, status, vabort);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[C::kBarOFull + so], tile_tx);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kOffO + so * C::kTile + b * 16384, &tm_do,
                        &bars[C::kBarOFull + so], 64 * b, w.kv * sh.g, qrow);
        }
      }
      if (!ok) {
        *vabort = 1;
        // drain this thread's own copies still in flight (the last issues of each ring)
        // (a Q tile may have been sent in the iteration whose O wait gave up)
        for (uint32_t it = q_sent > static_cast<uint32_t>(C::kNQ) ? q_sent - C::kNQ : 0u; it < q_sent; ++it)
          mbar_wait_ns(&bars[C::kBarQFull + it % C::kNQ], (it / C::kNQ) & 1u, 200000000ull);
        for (uint32_t it = qit > static_cast<uint32_t>(C::kNO) ? qit - C::kNO : 0u; it < qit; ++it)
          mbar_wait_ns(&bars[C::kBarOFull + it % C::kNO], (it / C::kNO) & 1u, 200000000ull);
        if (kv_pending) mbar_wait_ns(&bars[C::kBarKVFull], (uc) & 1u, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);
      const uint64_t dK0 = smem_desc(smem_u32(smem + C::kOffK), 16, 1024);
      const uint64_t dV0 = smem_desc(smem_u32(smem + C::kOffV), 16, 1024);
      const uint64_t dQk = smem_desc(smem_u32(smem + C::kOffQ), 16, 1024);     // K-major
      const uint64_t dQm = smem_desc(smem_u32(smem + C::kOffQ), 16384, 1024);  // MN-major
      const uint64_t dOk = smem_desc(smem_u32(smem + C::kOffO), 16, 1024);
      const uint64_t dOm = smem_desc(smem_u32(smem + C::kOffO), 16384, 1024);
      uint32_t qit = 0, uc = 0, n_s = 0, n_pds = 0;
      bool ok = true;
      // S^T = K Q^T for tile number it; waits for its Q and until the softmax has taken the
      // previous S out of TMEM
      auto issue_s = [&](uint32_t it) -> bool {
        const uint32_t sq = it % C::kNQ;
        if (!mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarQFull + sq], (it / C::kNQ) & 1u, status, vabort)) return false;
        if (n_s > 0 && !mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarSFree], (n_s - 1) & 1u, status, vabort))
          return false;
        tc_fence_after();
        const uint64_t q = dQk + static_cast<uint64_t>((sq * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(tmem + C::kColS, dK0 + o, q + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars[C::kBarSFull]);
        ++n_s;
        return true;
      };
      auto issue_dp = [&](uint32_t it) -> bool {
        const uint32_t so = it % C::kNO;
        if (!mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarOFull + so], (it / C::kNO) & 1u, status, vabort)) return false;
        tc_fence_after();
        const uint64_t o_ = dOk + static_cast<uint64_t>((so * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(tmem + C::kColDP, dV0 + o, o_ + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars[C::kBarDPFull]);
        return true;
      };
      // dV += P^T dO and dK += dS^T Q over the k-steps of P/dS chunk c (queries
      // 64 w + 32 c .. of both warpgroups w): kk = 2 c, 2 c + 1, 4 + 2 c, 5 + 2 c
      auto issue_acc = [&](uint32_t it, int c, bool acc) {
        const uint64_t q = dQm + static_cast<uint64_t>(((it % C::kNQ) * C::kTile) >> 4);
        const uint64_t o = dOm + static_cast<uint64_t>(((it % C::kNO) * C::kTile) >> 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = (i >> 1) * 4 + 2 * c + (i & 1);
          const uint64_t ko = static_cast<uint64_t>((kk * 2048) >> 4);
          const uint32_t pc = tmem + C::kColDP + packed_col(kk);
          mma_bf16_ts_w(tmem + C::kColDV, pc, o + ko, kIdAcc, (acc || i > 0) ? 1u : 0u);
          mma_bf16_ts_w(tmem + C::kColDK, pc + 16u, q + ko, kIdAcc, (acc || i > 0) ? 1u : 0u);
        }
        if (c == 1) {
          mma_commit_w(&bars[C::kBarQEmpty + it % C::kNQ]);
          mma_commit_w(&bars[C::kBarOEmpty + it % C::kNO]);
        }
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const KvUnit w = make_kv_unit<kPacked, kNoSuffix>(u, sh, vl);
        ok = mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarKVFull], uc & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        ok = issue_s(qit) && issue_dp(qit);
        for (int li = 0; li < w.n && ok; ++li) {
          const uint32_t it = qit + li;
          const bool more = li + 1 < w.n;
          if (more) {
            ok = issue_s(it + 1);
            if (!ok) break;
          }
          ok = mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarPDSFull], n_pds & 1u, status, vabort);
          if (!ok) break;
          if (li == 0 && uc > 0) {
            ok = mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarAccFree], (uc - 1) & 1u, status, vabort);
            if (!ok) break;
          }
          tc_fence_after();
          issue_acc(it, 0, li > 0);   // runs while the softmax finishes the second chunk
          ok = mbar_wait_hint<kHintDkdvMma>(&bars[C::kBarPDSFull + 1], n_pds & 1u, status, vabort);
          if (!ok) break;
          ++n_pds;
          tc_fence_after();
          issue_acc(it, 1, true);
          if (more) ok = issue_dp(it + 1);
        }
        if (!ok) break;
        qit += w.n;
        mma_commit_w(&bars[C::kBarAccDone]);
        if (u + static_cast<int>(gridDim.x) < n_units) mma_commit_w(&bars[C::kBarKVEmpty]);
      }
      if (!ok) *vabort = 1;
      mma_commit_w(&bars[C::kBarDrain]);
      mbar_wait_ns(&bars[C::kBarDrain], 0u, ok ? LS_WAIT_LIMIT_NS : 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // key within the tile (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = sh.scale * kLog2e;
    uint32_t qit = 0u, uc = 0u, n_tiles = 0u;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const KvUnit w = make_kv_unit<kPacked, kNoSuffix>(u, sh, vl);
      const int key = w.key0 + row;
      for (int li = 0; li < w.n; ++li, ++n_tiles) {
        // row statistics of this Q tile: every thread reads the same 1 KB (L1 broadcast)
        const float* rs = rowstats + (static_cast<int64_t>(w.kv) * n_qt + w.f0 + li) * 256;
        const float4* lse4 = reinterpret_cast<const float4*>(rs) + wg * 16;   // rows 64 wg ..
        const float4* dlt4 = reinterpret_cast<const float4*>(rs + 128) + wg * 16;
        // the next Q tile's row statistics (8 lines of 128 B) into L1 a step ahead, so that
        // its first reads do not wait on L2
        if (warp == 4 && lane < 8 && li + 1 < w.n) prefetch_l1(rs + 256 + lane * 32);
        ok = mbar_wait_hint<kHintDkdvSoftmax>(&bars[C::kBarSFull], n_tiles & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // ---- P^T from S^T (this warpgroup's 64 rows); S leaves TMEM first
        float p[64];
        {
          uint32_t sa[32], sb[32];
          tmem_ld32(lane_base + C::kColS + wg * 64, sa);
          tmem_ld32(lane_base + C::kColS + wg * 64 + 32, sb);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::kBarSFree]);
          // exponent arguments s c2 - LSE on fp32 pairs (one instruction per two queries)
          const uint64_t c2x2 = f2_pack(c2, c2);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 l4 = __ldg(lse4 + i);
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[4 * i + 0]), __uint_as_float(sa[4 * i + 1])),
                             c2x2, f2_pack(-l4.x, -l4.y)), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[4 * i + 2]), __uint_as_float(sa[4 * i + 3])),
                             c2x2, f2_pack(-l4.z, -l4.w)), x2, x3);
            p[4 * i + 0] = ex2_approx(x0);
            p[4 * i + 1] = ex2_approx(x1);
            p[4 * i + 2] = ex2_approx(x2);
            p[4 * i + 3] = ex2_approx(x3);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 l4 = __ldg(lse4 + 8 + i);
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sb[4 * i + 0]), __uint_as_float(sb[4 * i + 1])),
                             c2x2, f2_pack(-l4.x, -l4.y)), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sb[4 * i + 2]), __uint_as_float(sb[4 * i + 3])),
                             c2x2, f2_pack(-l4.z, -l4.w)), x2, x3);
            p[32 + 4 * i + 0] = ex2_approx(x0);
            p[32 + 4 * i + 1] = ex2_approx(x1);
            p[32 + 4 * i + 2] = ex2_approx(x2);
            p[32 + 4 * i + 3] = ex2_approx(x3);
          }
        }
        // causal suffix: rows r < lo of the tile see only suffix keys < this key
        if (!w.prompt) {
          const int v = sh.g * (key - (w.f0 + li - (kPacked ? vl.qt0[w.b] : 0)) * sh.qt);
          const int lo = v < 0 ? 0 : (v > 128 ? 128 : v);
          if (lo > wg * 64) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (wg * 64 + i < lo) p[i] = 0.0f;
          }
        }
        // ---- dS^T from dP^T; packed P^T / dS^T replace the fp32 dP^T chunk just read
        ok = mbar_wait_hint<kHintDkdvSoftmax>(&bars[C::kBarDPFull], (n_tiles & 1u), status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t dv[32];
          const uint32_t col = C::kColDP + wg * 64 + ch * 32;
          tmem_ld32(lane_base + col, dv);
          tmem_ld_wait();
          uint32_t pw[16], dw[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 d4 = __ldg(dlt4 + ch * 8 + i);
            const int c = ch * 32 + 4 * i;
            // dS = P (dP - Delta) on fp32 pairs
            float s0, s1, s2, s3;
            f2_unpack(f2_mul(f2_pack(p[c + 0], p[c + 1]),
                             f2_sub(f2_pack(__uint_as_float(dv[4 * i + 0]), __uint_as_float(dv[4 * i + 1])),
                                    f2_pack(d4.x, d4.y))), s0, s1);
            f2_unpack(f2_mul(f2_pack(p[c + 2], p[c + 3]),
                             f2_sub(f2_pack(__uint_as_float(dv[4 * i + 2]), __uint_as_float(dv[4 * i + 3])),
                                    f2_pack(d4.z, d4.w))), s2, s3);
            pw[2 * i] = pack_bf16x2(p[c + 0], p[c + 1]);
            pw[2 * i + 1] = pack_bf16x2(p[c + 2], p[c + 3]);
            dw[2 * i] = pack_bf16x2(s0, s1);
            dw[2 * i + 1] = pack_bf16x2(s2, s3);
          }
          tmem_st16(lane_base + col, pw);
          tmem_st16(lane_base + col + 16, dw);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::kBarPDSFull + ch]);
        }
      }
      if (!ok) break;
      qit += w.n;
      // epilogue: warpgroup 0 owns dV, warpgroup 1 owns dK
      ok = mbar_wait_hint<kHintDkdvSoftmax>(&bars[C::kBarAccDone], uc & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool valid = w.prompt ? (key < sh.P) : (key < w.R);
      const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
      const float mul = wg == 0 ? 1.0f : sh.scale;
      const int64_t off = ((static_cast<int64_t>(w.base) + key) * sh.Hkv + w.kv) * D;
      // fp32 accumulation: prompt keys, and suffix keys in block replay (rows P + key)
      const bool to_acc = w.prompt || suffix_to_acc != 0;
      const int64_t off_acc = w.prompt ? off : ((sh.P + key) * sh.Hkv + w.kv) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(lane_base + col + cc * 32, v);
        tmem_ld_wait();
        if (valid) {
          if (to_acc) {
            float4* dst = reinterpret_cast<float4*>((wg == 0 ? dv_acc : dk_acc) + off_acc + cc * 32);
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
  static constexpr int kTile = 128 * D * 2;         // Q, dO, K or V tile (128 rows)
  static constexpr int kNK = 3;                     // K ring: needed early (S) and late (dQ)
  static constexpr int kNV = 2;                     // V ring: needed by dP only
  static constexpr int kOffQ = 0, kOffDO = kTile, kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kNK * kTile;
  static constexpr int kOffBar = kOffV + kNV * kTile;
  static constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarQTmem = 2, kBarKFull = 3;
  static constexpr int kBarKEmpty = kBarKFull + kNK;
  static constexpr int kBarVFull = kBarKEmpty + kNK;
  static constexpr int kBarVEmpty = kBarVFull + kNV;
  static constexpr int kBarSFull = kBarVEmpty + kNV;
  static constexpr int kBarSFree = kBarSFull + 1;
  static constexpr int kBarDPFull = kBarSFree + 1;
  // dS written, per 32-column chunk of each warpgroup (chunk c: k-steps with bit 1 = c)
  static constexpr int kBarDSFull = kBarDPFull + 1;
  static constexpr int kBarDQDone = kBarDSFull + 2;
  static constexpr int kBarDQFree = kBarDQDone + 1;
  static constexpr int kBarDrain = kBarDQFree + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
  // TMEM: S at 0, dP at 128 (packed dS at packed_col(kk)), dQ at 256, and the unit's Q and
  // dO rows (bf16, the A operand of S = Q K^T and dP = dO V^T) at 384 and 384 + D/2.
  static constexpr uint32_t kColS = 0u, kColDP = 128u, kColDQ = 256u;
  static constexpr uint32_t kColQ = 384u, kColDO = 384u + D / 2;
};

struct QUnit {
  int kv;
  int f;       // flat 128-row Q tile over the packed responses
  int base;    // packed row of the response's first token
  int R;       // response length
  int t0;      // first query of the tile (response-local)
  int n_pt;    // prompt 128-key steps
  int n;       // total steps
};

// One response (base 0, length sh.R): flat unit u -> (kv head, 128-row Q tile).
__device__ __forceinline__ QUnit make_q_unit(int u, const AttnShape& sh, int n_qt) {
  QUnit w;
  w.kv = u / n_qt;
  w.f = u - w.kv * n_qt;
  w.base = 0;
  w.R = static_cast<int>(sh.R);
  w.t0 = w.f * sh.qt;
  int t_end = w.t0 + sh.qt;
  if (t_end > sh.R) t_end = static_cast<int>(sh.R);
  w.n_pt = static_cast<int>((sh.P + 127) / 128);
  w.n = w.n_pt + (t_end + 127) / 128;
  return w;
}

// Packed responses: flat unit u -> (kv head, flat Q tile f of response b).
__device__ __forceinline__ QUnit make_q_unit_packed(int u, const AttnShape& sh, const Varlen& vl) {
  QUnit w;
  const int n_qt = vl.qt0[vl.G];
  w.kv = u / n_qt;
  w.f = u - w.kv * n_qt;
  const int b = varlen_find(vl.qt0, vl.G, w.f);
  w.base = vl.row0[b];
  w.R = vl.row0[b + 1] - w.base;
  w.t0 = (w.f - vl.qt0[b]) * sh.qt;
  int t_end = w.t0 + sh.qt;
  if (t_end > w.R) t_end = w.R;
  w.n_pt = static_cast<int>((sh.P + 127) / 128);
  w.n = w.n_pt + (t_end + 127) / 128;
  return w;
}

template <bool kPacked, bool kNoSuffix>
__device__ __forceinline__ QUnit pick_q_unit(int u, const AttnShape& sh, int n_qt, const Varlen& vl) {
  if constexpr (kPacked) {
    return make_q_unit_packed(u, sh, vl);
  } else {
    QUnit w = make_q_unit(u, sh, n_qt);
    if constexpr (kNoSuffix) w.n = w.n_pt;
    return w;
  }
}

template <int D, bool kPacked, bool kNoSuffix>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_kp,
                       const __grid_constant__ CUtensorMap tm_vp,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do, const AttnShape sh,
                       const float* __restrict__ rowstats, uint16_t* __restrict__ dq,
                       const __grid_constant__ Varlen vl, uint32_t* status) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = kPacked ? vl.qt0[vl.G] : static_cast<int>((sh.R + sh.qt - 1) / sh.qt);
  const int n_units = sh.Hkv * n_qt;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[C::kBarQFull], 1);
    mbar_init(&bars[C::kBarQEmpty], 256);
    mbar_init(&bars[C::kBarQTmem], 256);
    for (int i = 0; i < C::kNK; ++i) {
      mbar_init(&bars[C::kBarKFull + i], 1);
      mbar_init(&bars[C::kBarKEmpty + i], 1);
    }
    for (int i = 0; i < C::kNV; ++i) {
      mbar_init(&bars[C::kBarVFull + i], 1);
      mbar_init(&bars[C::kBarVEmpty + i], 1);
    }
    mbar_init(&bars[C::kBarSFull], 1);
    mbar_init(&bars[C::kBarSFree], 256);
    mbar_init(&bars[C::kBarDPFull], 1);
    mbar_init(&bars[C::kBarDSFull], 256);
    mbar_init(&bars[C::kBarDSFull + 1], 256);
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
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      tma_prefetch_desc(&tm_vp);
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      uint32_t kit = 0, uc = 0, k_sent = 0;
      bool ok = true, q_sent = false;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const QUnit w = pick_q_unit<kPacked, kNoSuffix>(u, sh, n_qt, vl);
        q_sent = false;
        if (uc > 0) ok = mbar_wait_hint<kHintDqProducer>(&bars[C::kBarQEmpty], (uc - 1) & 1u, status, vabort);
        if (!ok) break;
        q_sent = true;
        mbar_arrive_expect_tx(&bars[C::kBarQFull],
                              static_cast<uint32_t>(2 * C::kBoxes * 128 * sh.g * sh.qt));
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(smem + C::kOffQ + b * 16384, &tm_q, &bars[C::kBarQFull], 64 * b,
                      w.kv * sh.g, (kPacked ? w.base : 0) + w.t0);
          tma_load_3d(smem + C::kOffDO + b * 16384, &tm_do, &bars[C::kBarQFull], 64 * b,
                      w.kv * sh.g, (kPacked ? w.base : 0) + w.t0);
        }
        for (int j = 0; j < w.n && ok; ++j, ++kit) {
          const bool pre = j < w.n_pt;
          const int key0 = pre ? 128 * j : (kPacked ? w.base : 0) + 128 * (j - w.n_pt);
          const uint32_t sk = kit % C::kNK, sv = kit % C::kNV;
          if (kit >= static_cast<uint32_t>(C::kNK))
            ok = mbar_wait_hint<kHintDqProducer>(&bars[C::kBarKEmpty + sk], ((kit / C::kNK) - 1) & 1u, status, vabort);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[C::kBarKFull + sk], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kOffK + sk * C::kTile + b * 16384, pre ? &tm_kp : &tm_ks,
                        &bars[C::kBarKFull + sk], 64 * b, w.kv, key0);
          ++k_sent;
          if (kit >= static_cast<uint32_t>(C::kNV))
            ok = mbar_wait_hint<kHintDqProducer>(&bars[C::kBarVEmpty + sv], ((kit / C::kNV) - 1) & 1u, status, vabort);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[C::kBarVFull + sv], C::kTile);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem + C::kOffV + sv * C::kTile + b * 16384, pre ? &tm_vp : &tm_vs,
                        &bars[C::kBarVFull + sv], 64 * b, w.kv, key0);
        }
      }
      if (!ok) {
        *vabort = 1;
        // drain this thread's own copies still in flight (a K tile may have been sent in the
        // iteration whose V wait gave up)
        for (uint32_t it = k_sent > static_cast<uint32_t>(C::kNK) ? k_sent - C::kNK : 0u; it < k_sent; ++it)
          mbar_wait_ns(&bars[C::kBarKFull + it % C::kNK], (it / C::kNK) & 1u, 200000000ull);
        for (uint32_t it = kit > static_cast<uint32_t>(C::kNV) ? kit - C::kNV : 0u; it < kit; ++it)
          mbar_wait_ns(&bars[C::kBarVFull + it % C::kNV], (it / C::kNV) & 1u, 200000000ull);
        if (q_sent) mbar_wait_ns(&bars[C::kBarQFull], uc & 1u, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);
      const uint64_t dKk = smem_desc(smem_u32(smem + C::kOffK), 16, 1024);      // K-major
      const uint64_t dKm = smem_desc(smem_u32(smem + C::kOffK), 16384, 1024);   // MN-major
      const uint64_t dVk = smem_desc(smem_u32(smem + C::kOffV), 16, 1024);
      uint32_t kit = 0, uc = 0, n_s = 0, n_ds = 0;
      bool ok = true;
      // S = Q K^T for key step number it; waits for its K and until the softmax has taken
      // the previous S out of TMEM
      auto issue_s = [&](uint32_t it) -> bool {
        const uint32_t sk = it % C::kNK;
        if (!mbar_wait_hint<kHintDqMma>(&bars[C::kBarKFull + sk], (it / C::kNK) & 1u, status, vabort)) return false;
        if (n_s > 0 && !mbar_wait_hint<kHintDqMma>(&bars[C::kBarSFree], (n_s - 1) & 1u, status, vabort))
          return false;
        tc_fence_after();
        const uint64_t k = dKk + static_cast<uint64_t>((sk * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ts_w(tmem + C::kColS, tmem + C::kColQ + kk * 8, k + o, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars[C::kBarSFull]);
        ++n_s;
        return true;
      };
      auto issue_dp = [&](uint32_t it) -> bool {
        const uint32_t sv = it % C::kNV;
        if (!mbar_wait_hint<kHintDqMma>(&bars[C::kBarVFull + sv], (it / C::kNV) & 1u, status, vabort)) return false;
        tc_fence_after();
        const uint64_t v = dVk + static_cast<uint64_t>((sv * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ts_w(tmem + C::kColDP, tmem + C::kColDO + kk * 8, v + o, kIdS,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bars[C::kBarDPFull]);
        mma_commit_w(&bars[C::kBarVEmpty + sv]);   // V is read by dP only
        return true;
      };
      // dQ += dS K over the k-steps of dS chunk c (keys 64 w + 32 c .. of both warpgroups w):
      // kk = 2 c, 2 c + 1, 4 + 2 c, 5 + 2 c
      auto issue_dq = [&](uint32_t it, int c, bool acc) {
        const uint32_t sk = it % C::kNK;
        const uint64_t k = dKm + static_cast<uint64_t>((sk * C::kTile) >> 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = (i >> 1) * 4 + 2 * c + (i & 1);
          mma_bf16_ts_w(tmem + C::kColDQ, tmem + C::kColDP + packed_col(kk),
                        k + static_cast<uint64_t>((kk * 2048) >> 4), kIdQ,
                        (acc || i > 0) ? 1u : 0u);
        }
        if (c == 1) mma_commit_w(&bars[C::kBarKEmpty + sk]);
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
        const QUnit w = pick_q_unit<kPacked, kNoSuffix>(u, sh, n_qt, vl);
        ok = mbar_wait_hint<kHintDqMma>(&bars[C::kBarQTmem], uc & 1u, status, vabort);
        if (!ok) break;
        tc_fence_after();
        ok = issue_s(kit) && issue_dp(kit);
        for (int j = 0; j < w.n && ok; ++j) {
          const uint32_t it = kit + j;
          const bool more = j + 1 < w.n;
          if (more) {
            ok = issue_s(it + 1);
            if (!ok) break;
          }
          ok = mbar_wait_hint<kHintDqMma>(&bars[C::kBarDSFull], n_ds & 1u, status, vabort);
          if (!ok) break;
          if (j == 0 && uc > 0) {
            ok = mbar_wait_hint<kHintDqMma>(&bars[C::kBarDQFree], (uc - 1) & 1u, status, vabort);
            if (!ok) break;
          }
          tc_fence_after();
          issue_dq(it, 0, j > 0);   // runs while the softmax finishes the second chunk
          ok = mbar_wait_hint<kHintDqMma>(&bars[C::kBarDSFull + 1], n_ds & 1u, status, vabort);
          if (!ok) break;
          ++n_ds;
          tc_fence_after();
          issue_dq(it, 1, true);
          if (more) ok = issue_dp(it + 1);
        }
        if (!ok) break;
        kit += w.n;
        mma_commit_w(&bars[C::kBarDQDone]);
      }
      if (!ok) *vabort = 1;
      mma_commit_w(&bars[C::kBarDrain]);
      mbar_wait_ns(&bars[C::kBarDrain], 0u, ok ? LS_WAIT_LIMIT_NS : 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = sh.scale * kLog2e;
    uint32_t uc = 0u, n_steps = 0u;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
      const QUnit w = pick_q_unit<kPacked, kNoSuffix>(u, sh, n_qt, vl);
      const int t = w.t0 + row / sh.g;
      const int hg = row % sh.g;
      const bool valid = (row < sh.g * sh.qt) && (kPacked ? t < w.R : t < sh.R);
      float lse2 = INFINITY, dlt = 0.0f;
      if (valid) {
        const float* rs = rowstats + (static_cast<int64_t>(w.kv) * n_qt + w.f) * 256;
        lse2 = rs[row];
        dlt = rs[128 + row];
      }
      // stage this unit's Q (warpgroup 0) or dO (warpgroup 1) row into TMEM; the previous
      // unit's MMAs have all completed (its dQ-done barrier was waited on)
      ok = mbar_wait_hint<kHintDqSoftmax>(&bars[C::kBarQFull], uc & 1u, status, vabort);
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
      for (int j = 0; j < w.n; ++j, ++n_steps) {
        ok = mbar_wait_hint<kHintDqSoftmax>(&bars[C::kBarSFull], n_steps & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // valid key columns of this row in this step
        int lim = 128;
        if (j < w.n_pt) {
          const int64_t rem = sh.P - 128ll * j;
          if (rem < 128) lim = static_cast<int>(rem);
        } else {
          const int v = t - 128 * (j - w.n_pt) + 1;
          lim = v < 0 ? 0 : (v > 128 ? 128 : v);
        }
        // ---- P from S (this warpgroup's 64 keys); S leaves TMEM first
        float p[64];
        {
          uint32_t sa[32], sb[32];
          tmem_ld32(lane_base + C::kColS + wg * 64, sa);
          tmem_ld32(lane_base + C::kColS + wg * 64 + 32, sb);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::kBarSFree]);
          // exponent arguments s c2 - LSE on fp32 pairs (one instruction per two keys)
          const uint64_t c2x2 = f2_pack(c2, c2), nl2 = f2_pack(-lse2, -lse2);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1, y0, y1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[2 * i]), __uint_as_float(sa[2 * i + 1])),
                             c2x2, nl2), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sb[2 * i]), __uint_as_float(sb[2 * i + 1])),
                             c2x2, nl2), y0, y1);
            p[2 * i] = ex2_approx(x0);
            p[2 * i + 1] = ex2_approx(x1);
            p[32 + 2 * i] = ex2_approx(y0);
            p[32 + 2 * i + 1] = ex2_approx(y1);
          }
        }
        if (lim < wg * 64 + 64) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (wg * 64 + i >= lim) p[i] = 0.0f;
        }
        // ---- dS from dP; packed dS replaces the fp32 dP chunk just read
        ok = mbar_wait_hint<kHintDqSoftmax>(&bars[C::kBarDPFull], n_steps & 1u, status, vabort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // both dP chunks are read with one wait (a single TMEM round trip)
        uint32_t dva[2][32];
        tmem_ld32(lane_base + C::kColDP + wg * 64, dva[0]);
        tmem_ld32(lane_base + C::kColDP + wg * 64 + 32, dva[1]);
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const uint32_t* dv = dva[ch];
          const uint32_t col = C::kColDP + wg * 64 + ch * 32;
          uint32_t dw[16];
          const uint64_t dlt2 = f2_pack(dlt, dlt);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // dS = P (dP - Delta) on fp32 pairs
            float s0, s1;
            f2_unpack(f2_mul(f2_pack(p[ch * 32 + 2 * i], p[ch * 32 + 2 * i + 1]),
                             f2_sub(f2_pack(__uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1])),
                                    dlt2)), s0, s1);
            dw[i] = pack_bf16x2(s0, s1);
          }
          tmem_st16(lane_base + col, dw);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::kBarDSFull + ch]);
        }
      }
      if (!ok) break;
      // epilogue: dQ * s -> bf16; warpgroup 0 stores columns [0, D/2), warpgroup 1 the rest
      ok = mbar_wait_hint<kHintDqSoftmax>(&bars[C::kBarDQDone], uc & 1u, status, vabort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int h = w.kv * sh.g + hg;
      uint16_t* drow = dq + ((kPacked ? static_cast<int64_t>(w.base) + t : static_cast<int64_t>(t)) * sh.Hq + h) * D;
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

template <int D, bool kPacked, bool kNoSuffix = false>
cudaError_t launch_dkdv_d(const BwdArgs& a, cudaStream_t s) {
  using C = DkdvCfg<D>;
  // the shared-memory opt-in is per device: remember it per device index
  static bool attr_set[kMaxDeviceCache] = {};
  const int dev = cached_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, kPacked, kNoSuffix>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t n_units =
      static_cast<int64_t>(a.sh.Hkv) * ((a.sh.P + 127) / 128 + (kNoSuffix ? 0 : a.vl.kt0[a.vl.G]));
  int grid = num_sms();
  if (n_units < grid) grid = static_cast<int>(n_units);
  attn_bwd_dkdv_kernel<D, kPacked, kNoSuffix><<<grid, kThreads, C::kSmem, s>>>(
      *a.tm_kp, *a.tm_vp, a.tm_ks, a.tm_vs, a.tm_q, a.tm_do, a.sh, a.rowstats, a.dk_acc,
      a.dv_acc, a.dk_suf, a.dv_suf, a.suffix_to_acc, a.vl, a.status);
  return cudaGetLastError();
}

template <int D, bool kPacked, bool kNoSuffix = false>
cudaError_t launch_dq_d(const BwdArgs& a, cudaStream_t s) {
  using C = DqCfg<D>;
  // the shared-memory opt-in is per device: remember it per device index
  static bool attr_set[kMaxDeviceCache] = {};
  const int dev = cached_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, kPacked, kNoSuffix>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t n_units = static_cast<int64_t>(a.sh.Hkv) * a.vl.qt0[a.vl.G];
  int grid = num_sms();
  if (n_units < grid) grid = static_cast<int>(n_units);
  attn_bwd_dq_kernel<D, kPacked, kNoSuffix><<<grid, kThreads, C::kSmem, s>>>(*a.tm_kp, *a.tm_vp, a.tm_ks, a.tm_vs,
                                                        a.tm_q, a.tm_do, a.sh, a.rowstats, a.dq,
                                                        a.vl, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  if (a.no_suffix) return a.sh.D == 128 ? launch_dkdv_d<128, false, true>(a, s) : launch_dkdv_d<64, false, true>(a, s);
  if (a.vl.G > 1) return a.sh.D == 128 ? launch_dkdv_d<128, true>(a, s) : launch_dkdv_d<64, true>(a, s);
  return a.sh.D == 128 ? launch_dkdv_d<128, false>(a, s) : launch_dkdv_d<64, false>(a, s);
}

cudaError_t launch_attn_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  if (a.no_suffix) return a.sh.D == 128 ? launch_dq_d<128, false, true>(a, s) : launch_dq_d<64, false, true>(a, s);
  if (a.vl.G > 1) return a.sh.D == 128 ? launch_dq_d<128, true>(a, s) : launch_dq_d<64, true>(a, s);
  return a.sh.D == 128 ? launch_dq_d<128, false>(a, s) : launch_dq_d<64, false>(a, s);
}

}  // namespace ls
