// fa_bwd_kernel.cuh -- attention backward from the saved LSE, for sm_103a.
//
// "Online Softmax 算法详解" section 8.3: the backward recomputes S = Q K^T,
// restores P = exp(scale S - LSE) from the LSE the forward saved (no second
// online softmax), and forms the gradients.  Written out (the derivative of
// O = softmax(scale S) V):
//   dV_j = sum_i P_ij dO_i          dP_ij = <dO_i, V_j>        D_i = <dO_i, O_i>
//   dS_ij = P_ij (dP_ij - D_i)      dK_j = scale sum_i dS_ij Q_i
//   dQ_i = scale sum_j dS_ij K_j
// A row whose LSE is -inf (no visible key) has P = 0 (section 7.3).
//
// Two kernels, no atomics (dQ would otherwise need fp32 reductions from every
// key tile of a head):
//   fa_bwd_dkdv_kernel  one 128-key tile per CTA, K_j and V_j in shared memory,
//     looping over the query tiles that see it, each as two half-steps of 64
//     queries.  S^T = K_j Q^T and dP^T = V_j dO^T of a half-step go to TMEM
//     buffer b (two buffers of 64 + 64 columns, then dV and dK: 512 columns at
//     d = 128); compute warpgroup b owns buffer b (queries [64b, 64b + 64) of
//     every tile): thread t owns key t (TMEM lane t) and writes P^T and dS^T
//     (bf16 pairs) back into the columns it has just read; dV_j += P^T dO and
//     dK_j += dS^T Q then take them as the TMEM A operand.  P^T is released
//     on its own, before dS^T is formed, so dV (and after it the next S^T of
//     the buffer) overlaps the second half of the warpgroup's work.  The MMA warp issues
//     dV, dK of half-step h, then S^T of h+2 once dV(h) is done and dP^T of h+2
//     once dK(h) is done: each follows the previous MMA on the tensor pipe, and
//     each warpgroup has two half-steps of MMA time for its exponentials.
//   fa_bwd_dq_kernel  one 128-row query tile per CTA, Q_i and dO_i in shared
//     memory, looping over the key tiles it sees: S = Q_i K_j^T and
//     dP = dO_i V_j^T, each released as soon as every row has read it, dS
//     (bf16) into one of two TMEM buffers of its own, and dQ_i += dS K_j.
//   S and dP are recomputed by both: 7 MMAs per tile pair instead of 5.
// fa_bwd_pre_kernel  -D_i and -LSE * log2(e) per row (-inf for a row with no
//   visible key or past Nq, so exp2(S c + nlse2) is exactly 0 there), padded
//   to whole 128-row tiles so the kernels copy them in 512-byte pieces; stored
//   negated so P and dS take packed two-lane FMA / add / multiply directly.
//
// In the dQ kernel the two compute warpgroups split the 128 columns of S / dP:
// warpgroup h takes columns [64h, 64h + 64) and writes its bf16 pairs into
// columns [32h, 32h + 32) of the dS buffer, so the buffer holds keys in order
// and the A operand's K-slice kk (16 keys) is at column 8 kk.
//
// Every wait is bounded (fa_wait.cuh); a wait that runs out stops the CTA
// without writing its outputs.
#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_wait.cuh"

namespace fa {

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kRows = 128;               // rows of a Q / K / V / dO tile
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) swizzle chunks
  static constexpr int kChunkBytes = kRows * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kVecBytes = kRows * 4;     // nlse2 or nd of one tile
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kStageBytesA = 2 * kTileBytes + 2 * kVecBytes;  // Q_i, dO_i, nlse2, nd
  // dQ kernel: K_j and V_j in separate slots of a ring, K_j at position 2 j
  // and V_j at 2 j + 1; each slot is released by its own last reader.
  static constexpr int kSlotsFit = (227 * 1024 - 1024 - 2 * kTileBytes - 1024) / kTileBytes;
  static constexpr int kSlotsB = kSlotsFit > 8 ? 8 : kSlotsFit;
  static constexpr int kStageBytesB = kTileBytes;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kSmemA = 1024 + 2 * kTileBytes + kStages * kStageBytesA + kCtlBytes;
  static constexpr int kSmemB = 1024 + 2 * kTileBytes + kSlotsB * kStageBytesB + kCtlBytes;
  static_assert(kSlotsB >= 4, "dQ kernel ring");
  static_assert(kSmemA <= 227 * 1024 && kSmemB <= 227 * 1024, "shared memory");
  static_assert(kStageBytesA % 1024 == 0, "stage alignment");
  static constexpr int kThreads = 384;  // two compute warpgroups + load / MMA / alloc warps
  // Two MMA issuers: one for the products that fill S / dP, one for the
  // products that consume P / dS (dK/dV kernel: dV, dK; dQ kernel: dQ).
  static constexpr int kLoadWarp = 8, kMmaWarp = 9, kAllocWarp = 10, kMmaWarp2 = 11;
  // dK/dV kernel registers: launched with 168 per thread, then setmaxnreg
  // moves them to the compute warpgroups (the split adds up to the launch
  // budget, or setmaxnreg.inc could never be granted).
  static constexpr int kRegLaunchA = 168, kRegComputeA = 216, kRegOtherA = 72;
  static_assert(2 * kRegComputeA + kRegOtherA == 3 * kRegLaunchA, "setmaxnreg split");
  static constexpr int kTmemCols = 512;
  // dK/dV kernel: S^T / P^T buffers at 64 b, dP^T / dS^T at 128 + 64 b, then
  // the two accumulators.
  static constexpr int kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
  // dQ kernel: S, dP, two bf16 dS buffers of 64 columns, dQ.
  static constexpr int kDPq = 128, kDS0 = 256, kDQ = 384;
};

struct __align__(8) BwdCtl {
  uint64_t fixed_full;  // K_j, V_j (dK/dV) or Q_i, dO_i (dQ) landed
  uint64_t full[8];     // ring stage / slot landed
  uint64_t empty[8];    // every MMA reading the stage / slot completed
  uint64_t s_full[2];   // S(^T) of this step in TMEM (dK/dV: per buffer)
  uint64_t s_free;      // dQ kernel: S read by all 256 compute threads
  uint64_t dp_free;     // dQ kernel: dP read by all 256 compute threads
  uint64_t dp_full[2];  // dP(^T) in TMEM (buffer)
  uint64_t ready[2];    // bf16 P^T (dK/dV kernel) or dS (dQ kernel) written back to TMEM
  uint64_t ds_ready[2]; // dK/dV kernel: bf16 dS^T written back to TMEM
  uint64_t done_a[2];   // dK/dV kernel: dV MMA of a buffer done (its S columns free)
  uint64_t done_b[2];   // dK MMA of a buffer done (dP columns free) / dQ MMA of a buffer done
  uint64_t drain;       // every MMA of the CTA completed
  uint32_t tmem_base;
  int abort;
};

// Masks: key k is visible to query q iff q + off - wl <= k <= q + off + wr
// (off = Nk - Nq, -1 = open side).
__device__ __forceinline__ bool bwd_visible(int q, int k, const BwdParams& p) {
  const int qa = q + p.Nk - p.Nq;
  return (p.wl < 0 || k >= qa - p.wl) && (p.wr < 0 || k <= qa + p.wr) && k < p.Nk;
}

// Every (query, key) pair of the 128 x 128 tile pair is visible (a test that
// is the same for every thread, so the mask loop is skipped as a whole).
__device__ __forceinline__ bool bwd_tile_all_visible(int q0, int key0, const BwdParams& p) {
  const int off = p.Nk - p.Nq;
  const int q_last = min(q0 + 127, p.Nq - 1);
  const int k_last = key0 + 127;
  return k_last < p.Nk && (p.wl < 0 || key0 >= q_last + off - p.wl) &&
         (p.wr < 0 || k_last <= q0 + off + p.wr);
}

// Shared-memory descriptors of a [128 rows][D] bf16 tile (128-byte swizzle):
// as a K-major operand (K = D) and as an MN-major B operand (N = D, K = rows).
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return smem_desc_sw128(saddr, 16, 1024);
}
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  return smem_desc_sw128(saddr, BwdCfg<D>::kChunkBytes, 1024);
}
// K-slice kk (16 elements) of a K-major tile: chunk kk / 4, 32 bytes per slice.
template <int D>
__device__ __forceinline__ uint32_t kslice_kmajor(int kk) {
  return static_cast<uint32_t>((kk / 4) * BwdCfg<D>::kChunkBytes + (kk % 4) * 32) >> 4;
}
// K-slice kk (16 rows) of an MN-major tile: two 8-row groups of 1024 bytes.
__device__ __forceinline__ uint32_t kslice_mnmajor(int kk) {
  return static_cast<uint32_t>(kk * 2048) >> 4;
}
// Stage a [128][D] bf16 tile row for a TMA store: row t, columns
// [c0, c0 + 32) (packed pairs w[16]) into the 128-byte-swizzled layout.
template <int D>
__device__ __forceinline__ void stage_row32(uint32_t tile, int t, int c0, const uint32_t* w) {
  const int chunk = c0 / 64;
  const int u0 = (c0 % 64) / 8;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = u0 + q;
    st_shared_v4(tile + chunk * BwdCfg<D>::kChunkBytes + t * 128 + ((u ^ (t & 7)) << 4), w[4 * q],
                 w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// ===================================================================== dK, dV
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::kTileBytes;
  uint8_t* sRing = sV + C::kTileBytes;  // stage: Q_i, dO_i, nlse2[128], nd[128]
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sRing + C::kStages * C::kStageBytesA);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = blockIdx.x;  // key tile
  const int bh = blockIdx.y;
  const int key0 = kt * C::kRows;
  const int off = p.Nk - p.Nq;
  // query tiles with a row that sees a key of this tile
  const int k_last = min(key0 + C::kRows, p.Nk) - 1;
  const int qlo = p.wr < 0 ? 0 : max(0, key0 - off - p.wr);
  const int qhi = p.wl < 0 ? p.Nq - 1 : min(p.Nq - 1, k_last - off + p.wl);
  const int i_lo = qlo / C::kRows;
  const int n = qhi >= qlo ? qhi / C::kRows + 1 - i_lo : 0;

  const uint32_t bar_fixed = smem_u32(&ctl->fixed_full);
  const uint32_t bar_full = smem_u32(&ctl->full[0]);
  const uint32_t bar_empty = smem_u32(&ctl->empty[0]);
  // per buffer b: + 8 b
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_dp = smem_u32(&ctl->dp_full[0]);
  const uint32_t bar_ready = smem_u32(&ctl->ready[0]);
  const uint32_t bar_dsr = smem_u32(&ctl->ds_ready[0]);
  const uint32_t bar_dv = smem_u32(&ctl->done_a[0]);
  const uint32_t bar_dk = smem_u32(&ctl->done_b[0]);
  const uint32_t bar_drain = smem_u32(&ctl->drain);

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s + 8 * b, 1);
      mbar_init(bar_dp + 8 * b, 1);
      mbar_init(bar_ready + 8 * b, 128);
      mbar_init(bar_dsr + 8 * b, 128);
      mbar_init(bar_dv + 8 * b, 1);
      mbar_init(bar_dk + 8 * b, 1);
    }
    mbar_init(bar_drain, 2);  // one commit per MMA issuer
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kAllocWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const WaitCtx wc{&ctl->abort, p.status, p.timeout_ns};

  if (warp >= 8) {
   setmaxnreg_dec<C::kRegOtherA>();
   if (warp == C::kLoadWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      // (n = 0: no query sees this key tile; nothing is loaded, dK = dV = 0)
      if (n > 0) {
        mbar_arrive_expect_tx(bar_fixed, 2 * C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(smem_u32(sK + c * C::kChunkBytes), &tm_k, bar_fixed, c * 64, key0, bh);
          tma_load_3d(smem_u32(sV + c * C::kChunkBytes), &tm_v, bar_fixed, c * 64, key0, bh);
        }
      }
      const uint64_t pol = l2_policy_evict_last();
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      for (int s = 0; ok && s < n; ++s) {
        const int st = s % C::kStages, use = s / C::kStages;
        if (use > 0 && !wait_bounded(bar_empty + 8 * st, (use - 1) & 1, wc)) {
          ok = false;
          break;
        }
        const int q0 = (i_lo + s) * C::kRows;
        uint8_t* base = sRing + st * C::kStageBytesA;
        const uint32_t full = bar_full + 8 * st;
        mbar_arrive_expect_tx(full, 2 * C::kTileBytes + 2 * C::kVecBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(smem_u32(base + c * C::kChunkBytes), &tm_q, full, c * 64, q0, bh);
          tma_load_3d(smem_u32(base + C::kTileBytes + c * C::kChunkBytes), &tm_do, full, c * 64, q0,
                      bh);
        }
        const size_t vrow = static_cast<size_t>(bh) * p.nq_pad + q0;
        bulk_load(smem_u32(base + 2 * C::kTileBytes), p.nlse2 + vrow, C::kVecBytes, full, pol);
        bulk_load(smem_u32(base + 2 * C::kTileBytes + C::kVecBytes), p.nd + vrow, C::kVecBytes,
                  full, pol);
        issued_mask |= 1u << st;
        issued_par = (issued_par & ~(1u << st)) | (static_cast<uint32_t>(use & 1) << st);
      }
      for (int s = 0; s < C::kStages; ++s)
        if ((issued_mask >> s) & 1u) wait_own(bar_full + 8 * s, (issued_par >> s) & 1u, p.timeout_ns);
      if (n > 0) wait_own(bar_fixed, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp2) {
    // --------------------------------------------------------- MMA issuers
    // Half-step hs = 2 s + b covers queries [64 b, 64 b + 64) of query tile
    // s and uses TMEM buffer b.  Warp kMmaWarp2 fills buffers (S^T, dP^T);
    // warp kMmaWarp consumes them (dV, dK).  Between the two only barriers:
    // S^T of hs+2 once dV of hs has read P^T, dP^T once dK has read dS^T.
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false);  // A = K or V, B = Q or dO rows (K-major)
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, true);  // B = dO or Q rows (MN-major)
    const int nh = 2 * n;
    auto stage_base = [&](int hs) {
      return smem_u32(sRing + ((hs >> 1) % C::kStages) * C::kStageBytesA);
    };
    bool ok = n > 0 && warp_wait(bar_fixed, 0, wc);
    if (warp == C::kMmaWarp2) {
      const uint64_t dK = desc_kmajor<D>(smem_u32(sK));
      const uint64_t dV = desc_kmajor<D>(smem_u32(sV));
      // S^T = K_j Q_h^T into buffer hs & 1 (Q_h: 64 rows, 8 KB into every chunk)
      auto issue_s = [&](int hs) {
        const uint64_t dQk = desc_kmajor<D>(stage_base(hs) + (hs & 1) * 64 * 128);
        const uint32_t dst = tmem + C::kS + 64 * (hs & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss_elect(dst, dK + kslice_kmajor<D>(kk), dQk + kslice_kmajor<D>(kk), kIdescS, kk > 0);
        mma_commit_elect(bar_s + 8 * (hs & 1));
      };
      auto issue_dp = [&](int hs) {  // dP^T = V_j dO_h^T
        const uint64_t dOk = desc_kmajor<D>(stage_base(hs) + C::kTileBytes + (hs & 1) * 64 * 128);
        const uint32_t dst = tmem + C::kDP + 64 * (hs & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss_elect(dst, dV + kslice_kmajor<D>(kk), dOk + kslice_kmajor<D>(kk), kIdescS, kk > 0);
        mma_commit_elect(bar_dp + 8 * (hs & 1));
      };
      if (ok) ok = warp_wait(bar_full, 0, wc);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
        issue_s(1);
        issue_dp(1);
      }
      for (int hs = 0; ok && hs + 2 < nh; ++hs) {
        const int b = hs & 1, nx = hs + 2;
        const uint32_t par = static_cast<uint32_t>((hs >> 1) & 1);
        if (b == 0) ok = warp_wait(bar_full + 8 * ((nx >> 1) % C::kStages), ((nx >> 1) / C::kStages) & 1, wc);
        ok = ok && warp_wait(bar_dv + 8 * b, par, wc);
        if (!ok) break;
        tc_fence_after();
        issue_s(nx);
        ok = warp_wait(bar_dk + 8 * b, par, wc);
        if (!ok) break;
        tc_fence_after();
        issue_dp(nx);
      }
    } else {
      for (int hs = 0; ok && hs < nh; ++hs) {
        const int b = hs & 1;
        ok = warp_wait(bar_ready + 8 * b, static_cast<uint32_t>((hs >> 1) & 1), wc);
        if (!ok) break;
        tc_fence_after();
        const uint32_t base = stage_base(hs);
        const uint64_t dOmn = desc_mnmajor<D>(base + C::kTileBytes);
        const uint64_t dQmn = desc_mnmajor<D>(base);
        const uint32_t pa = tmem + C::kS + 64 * b, da = tmem + C::kDP + 64 * b;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dV += P^T dO_h (K = 64 queries: rows 64 b + 16 kk)
          mma_bf16_ts_elect(tmem + C::kDV, pa + 8 * kk, dOmn + kslice_mnmajor(4 * b + kk), kIdescAcc,
                            (hs > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(bar_dv + 8 * b);
        ok = warp_wait(bar_dsr + 8 * b, static_cast<uint32_t>((hs >> 1) & 1), wc);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dK += dS^T Q_h
          mma_bf16_ts_elect(tmem + C::kDK, da + 8 * kk, dQmn + kslice_mnmajor(4 * b + kk), kIdescAcc,
                            (hs > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(bar_dk + 8 * b);
        // both halves of the tile done: S^T / dP^T (the other warp) completed
        // before their P^T / dS^T were written back, so this commit covers
        // every read of the stage
        if (b == 1) mma_commit_elect(bar_empty + 8 * ((hs >> 1) % C::kStages));
      }
    }
    // everything issued completes before the epilogue reads TMEM / TMEM is freed
    mma_commit_elect(bar_drain);
    if (n > 0) wait_own(bar_drain, 0, p.timeout_ns);
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<C::kRegComputeA>();
    // ------------------------------------------------ compute warpgroups
    const int h = warp >> 2;               // buffer / query half of every tile
    const int t = (warp & 3) * 32 + lane;  // key row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int key = key0 + t;
    const float c = p.scale_log2;
    const uint32_t tS = tmem + lane_off + C::kS + 64 * h;
    const uint32_t tDP = tmem + lane_off + C::kDP + 64 * h;
    bool ok = true;
    for (int s = 0; ok && s < n; ++s) {
      const int st = s % C::kStages;
      const int q0 = (i_lo + s) * C::kRows + 64 * h;  // this half's first query
      const float* nlv = reinterpret_cast<const float*>(sRing + st * C::kStageBytesA + 2 * C::kTileBytes) + 64 * h;
      const float* ndv = nlv + C::kRows;
      // P^T first, from S^T alone, so dV += P^T dO (and S^T of half-step
      // h + 2 after it) can start while dS^T is still being formed.  The
      // stage's own barrier makes the bulk-copied nlse2 / nd visible here.
      ok = warp_wait(bar_full + 8 * st, (s / C::kStages) & 1, wc) && warp_wait(bar_s + 8 * h, s & 1, wc);
      if (!ok) break;
      tc_fence_after();
      const bool all_vis = bwd_tile_all_visible(q0, key0, p);  // (a superset test: 128 queries)
      float pv[64];
      {
        uint32_t srow[64];
        tmem_ld64_sync(tS, srow);
        const uint64_t c2 = f2_pack(c, c);
#pragma unroll
        for (int k = 0; k < 64; k += 4) {  // 2^(S c - LSE log2 e), two lanes per FMA
          const float4 a4 = *reinterpret_cast<const float4*>(nlv + k);
          float x0, x1, x2, x3;
          f2_unpack(ffma2(f2_pack(__uint_as_float(srow[k]), __uint_as_float(srow[k + 1])), c2,
                          f2_pack(a4.x, a4.y)), x0, x1);
          f2_unpack(ffma2(f2_pack(__uint_as_float(srow[k + 2]), __uint_as_float(srow[k + 3])), c2,
                          f2_pack(a4.z, a4.w)), x2, x3);
          pv[k] = ex2_approx(x0);
          pv[k + 1] = ex2_approx(x1);
          pv[k + 2] = ex2_approx(x2);
          pv[k + 3] = ex2_approx(x3);
        }
      }
      // edge tiles only: the mask in a block of its own, so fully visible
      // tiles run the loop above with no per-element test
      if (!all_vis) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (!bwd_visible(q0 + k, key, p)) pv[k] = 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack_bf16x2(pv[2 * k], pv[2 * k + 1]);
        tmem_st32(tS, pk);  // pairs into columns already read: [0, 32)
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ready + 8 * h);
      // dS^T = P^T (dP^T - D) once dP^T has landed
      if (!warp_wait(bar_dp + 8 * h, s & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t drow[64];
        tmem_ld64_sync(tDP, drow);
        uint32_t dk[32];
#pragma unroll
        for (int k = 0; k < 64; k += 4) {  // P (dP - D), two lanes per add / multiply
          const float4 d4 = *reinterpret_cast<const float4*>(ndv + k);
          float y0, y1, y2, y3;
          f2_unpack(fmul2(f2_pack(pv[k], pv[k + 1]),
                          fadd2(f2_pack(__uint_as_float(drow[k]), __uint_as_float(drow[k + 1])),
                                f2_pack(d4.x, d4.y))), y0, y1);
          f2_unpack(fmul2(f2_pack(pv[k + 2], pv[k + 3]),
                          fadd2(f2_pack(__uint_as_float(drow[k + 2]), __uint_as_float(drow[k + 3])),
                                f2_pack(d4.z, d4.w))), y2, y3);
          dk[k >> 1] = pack_bf16x2(y0, y1);
          dk[(k >> 1) + 1] = pack_bf16x2(y2, y3);
        }
        tmem_st32(tDP, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_dsr + 8 * h);
    }
    // ---- epilogue: dV, dK (x scale) -> bf16 -> the K / V buffers -> TMA store
    if (ok && n > 0) ok = warp_wait(bar_drain, 0, wc);
    const bool bad = named_bar_or(1, 256, !ok || *wc.abort);
    if (!bad) {
      if (n > 0) tc_fence_after();
      const uint32_t stK = smem_u32(sK), stV = smem_u32(sV);
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // 0: dV, 1: dK
        const float mul = part ? p.scale : 1.f;
        const uint32_t src = tmem + lane_off + (part ? C::kDK : C::kDV);
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 32) {
          const int col = h * (D / 2) + cc;
          uint32_t r[32];
          if (n > 0) {
            tmem_ld32_sync(src + col, r);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(__uint_as_float(r[2 * k]) * mul, __uint_as_float(r[2 * k + 1]) * mul);
          stage_row32<D>(part ? stK : stV, t, col, w);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int ch = 0; ch < C::kChunks; ++ch) {
          tma_store_3d(&tm_dk, stK + ch * C::kChunkBytes, ch * 64, key0, bh);
          tma_store_3d(&tm_dv, stV + ch * C::kChunkBytes, ch * 64, key0, bh);
        }
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kAllocWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ========================================================================= dQ
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* sQ = smem;
  uint8_t* sDO = sQ + C::kTileBytes;
  uint8_t* sRing = sDO + C::kTileBytes;  // slots: K_j at position 2 j, V_j at 2 j + 1
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sRing + C::kSlotsB * C::kStageBytesB);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = p.causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int q0 = qt * C::kRows;
  const int off = p.Nk - p.Nq;
  // key tiles holding a key some row of this tile sees
  const int q_last = min(q0 + C::kRows, p.Nq) - 1;
  const int klo = p.wl < 0 ? 0 : max(0, q0 + off - p.wl);
  const int khi = p.wr < 0 ? p.Nk - 1 : min(p.Nk - 1, q_last + off + p.wr);
  const int j_lo = klo / C::kRows;
  const int n = khi >= klo ? khi / C::kRows + 1 - j_lo : 0;

  const uint32_t bar_fixed = smem_u32(&ctl->fixed_full);
  const uint32_t bar_full = smem_u32(&ctl->full[0]);
  const uint32_t bar_empty = smem_u32(&ctl->empty[0]);
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_sfree = smem_u32(&ctl->s_free);
  const uint32_t bar_dp = smem_u32(&ctl->dp_full[0]);
  const uint32_t bar_dpfree = smem_u32(&ctl->dp_free);
  const uint32_t bar_ready = smem_u32(&ctl->ready[0]);    // + 8 b
  const uint32_t bar_dq = smem_u32(&ctl->done_b[0]);      // + 8 b
  const uint32_t bar_drain = smem_u32(&ctl->drain);

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kSlotsB; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 256);
    mbar_init(bar_dp, 1);
    mbar_init(bar_dpfree, 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_ready + 8 * b, 256);
      mbar_init(bar_dq + 8 * b, 1);
    }
    mbar_init(bar_drain, 2);  // one commit per MMA issuer
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kAllocWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const WaitCtx wc{&ctl->abort, p.status, p.timeout_ns};

  if (warp == C::kLoadWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      if (n > 0) {
        mbar_arrive_expect_tx(bar_fixed, 2 * C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(smem_u32(sQ + c * C::kChunkBytes), &tm_q, bar_fixed, c * 64, q0, bh);
          tma_load_3d(smem_u32(sDO + c * C::kChunkBytes), &tm_do, bar_fixed, c * 64, q0, bh);
        }
      }
      uint32_t issued_mask = 0, issued_par = 0;
      for (int pos = 0; pos < 2 * n; ++pos) {
        const int sl = pos % C::kSlotsB, use = pos / C::kSlotsB;
        if (use > 0 && !wait_bounded(bar_empty + 8 * sl, (use - 1) & 1, wc)) break;
        const int k0 = (j_lo + (pos >> 1)) * C::kRows;
        uint8_t* base = sRing + sl * C::kStageBytesB;
        const uint32_t full = bar_full + 8 * sl;
        const CUtensorMap* map = (pos & 1) ? &tm_v : &tm_k;
        mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(base + c * C::kChunkBytes), map, full, c * 64, k0, bh);
        issued_mask |= 1u << sl;
        issued_par = (issued_par & ~(1u << sl)) | (static_cast<uint32_t>(use & 1) << sl);
      }
      for (int s = 0; s < C::kSlotsB; ++s)
        if ((issued_mask >> s) & 1u) wait_own(bar_full + 8 * s, (issued_par >> s) & 1u, p.timeout_ns);
      if (n > 0) wait_own(bar_fixed, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp2) {
    // --------------------------------------------------------- MMA issuers
    // Warp kMmaWarp: S(j) = Q_i K_j^T once every row has read S(j-1), and
    // dP(j) = dO_i V_j^T once every row has read dP(j-1).
    // Warp kMmaWarp2: dQ += dS(j) K_j once dS(j) is in its TMEM buffer j & 1.
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, true);  // B = K_j (MN-major)
    auto slot = [&](int pos) { return smem_u32(sRing + (pos % C::kSlotsB) * C::kStageBytesB); };
    auto slot_full = [&](int pos) {
      return warp_wait(bar_full + 8 * (pos % C::kSlotsB), (pos / C::kSlotsB) & 1, wc);
    };
    bool ok = n > 0 && warp_wait(bar_fixed, 0, wc);
    if (warp == C::kMmaWarp) {
      const uint64_t dQk = desc_kmajor<D>(smem_u32(sQ));
      const uint64_t dOk = desc_kmajor<D>(smem_u32(sDO));
      for (int j = 0; ok && j < n; ++j) {
        ok = slot_full(2 * j) && (j == 0 || warp_wait(bar_sfree, (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t dKk = desc_kmajor<D>(slot(2 * j));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss_elect(tmem + C::kS, dQk + kslice_kmajor<D>(kk), dKk + kslice_kmajor<D>(kk),
                              kIdescS, kk > 0);
          mma_commit_elect(bar_s);
        }
        ok = slot_full(2 * j + 1) && (j == 0 || warp_wait(bar_dpfree, (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t dVk = desc_kmajor<D>(slot(2 * j + 1));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss_elect(tmem + C::kDPq, dOk + kslice_kmajor<D>(kk), dVk + kslice_kmajor<D>(kk),
                              kIdescS, kk > 0);
          mma_commit_elect(bar_dp);
          mma_commit_elect(bar_empty + 8 * ((2 * j + 1) % C::kSlotsB));  // V_j read
        }
      }
    } else {
      for (int j = 0; ok && j < n; ++j) {
        ok = warp_wait(bar_ready + 8 * (j & 1), (j >> 1) & 1, wc);  // dS(j) written back
        if (!ok) break;
        tc_fence_after();
        const uint64_t dKmn = desc_mnmajor<D>(slot(2 * j));
        const uint32_t src = tmem + C::kDS0 + 64 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ += dS K_j (K = 128 keys, 8 columns per K-step)
          mma_bf16_ts_elect(tmem + C::kDQ, src + 8 * kk, dKmn + kslice_mnmajor(kk), kIdescDQ,
                            (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(bar_dq + 8 * (j & 1));
        // K_j: S(j) (the other warp) completed before dS(j) could exist
        mma_commit_elect(bar_empty + 8 * ((2 * j) % C::kSlotsB));
      }
    }
    mma_commit_elect(bar_drain);
    if (n > 0) wait_own(bar_drain, 0, p.timeout_ns);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------ compute warpgroups
    const int h = warp >> 2;
    const int t = (warp & 3) * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int row = q0 + t;
    const size_t vrow = static_cast<size_t>(bh) * p.nq_pad + row;
    const float c = p.scale_log2;
    const uint64_t nl2 = f2_pack(p.nlse2[vrow], p.nlse2[vrow]), nd2 = f2_pack(p.nd[vrow], p.nd[vrow]);
    const uint64_t c2 = f2_pack(c, c);
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const int key0 = (j_lo + j) * C::kRows;
      ok = warp_wait(bar_s, j & 1, wc);
      if (!ok) break;
      tc_fence_after();
      // this warpgroup's 64 keys of S; the buffer is released right away
      float pv[64];
      {
        uint32_t sr[64];
        tmem_ld64_sync(tmem + lane_off + C::kS + 64 * h, sr);
        tc_fence_before();
        mbar_arrive(bar_sfree);  // S may be overwritten by S of step j+1
#pragma unroll
        for (int k = 0; k < 64; k += 2) {  // 2^(S c - LSE log2 e), two lanes per FMA
          float x0, x1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nl2), x0, x1);
          pv[k] = ex2_approx(x0);
          pv[k + 1] = ex2_approx(x1);
        }
      }
      if (!bwd_tile_all_visible(q0, key0, p)) {  // edge tiles only
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (!bwd_visible(row, key0 + 64 * h + k, p)) pv[k] = 0.f;
      }
      ok = warp_wait(bar_dp, j & 1, wc);
      if (!ok) break;
      tc_fence_after();
      uint32_t dk[32];
      {
        uint32_t dr[64];
        tmem_ld64_sync(tmem + lane_off + C::kDPq + 64 * h, dr);
        tc_fence_before();
        mbar_arrive(bar_dpfree);  // dP may be overwritten by dP of step j+1
#pragma unroll
        for (int k = 0; k < 64; k += 2) {  // P (dP - D)
          float y0, y1;
          f2_unpack(fmul2(f2_pack(pv[k], pv[k + 1]),
                          fadd2(f2_pack(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1])), nd2)), y0, y1);
          dk[k >> 1] = pack_bf16x2(y0, y1);
        }
      }
      // dS buffer j & 1 is free once dQ += dS(j-2) K has completed
      if (j >= 2 && !warp_wait(bar_dq + 8 * (j & 1), ((j - 2) >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32(tmem + lane_off + C::kDS0 + 64 * (j & 1) + 32 * h, dk);  // keys 64 h .. 64 h + 63
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ready + 8 * (j & 1));
    }
    // ---- epilogue: dQ x scale -> bf16 -> the Q buffer -> TMA store
    if (ok && n > 0) ok = warp_wait(bar_drain, 0, wc);
    const bool bad = named_bar_or(1, 256, !ok || *wc.abort);
    if (!bad && q0 < p.Nq) {
      if (n > 0) tc_fence_after();
      const uint32_t stQ = smem_u32(sQ);
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        const int col = h * (D / 2) + cc;
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32_sync(tmem + lane_off + C::kDQ + col, r);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(r[2 * k]) * p.scale, __uint_as_float(r[2 * k + 1]) * p.scale);
        stage_row32<D>(stQ, t, col, w);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int ch = 0; ch < C::kChunks; ++ch)
          tma_store_3d(&tm_dq, stQ + ch * C::kChunkBytes, ch * 64, q0, bh);
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kAllocWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================ preprocess
// nd_i = -<dO_i, O_i> (fp32 over bf16 inputs) and nlse2_i = -LSE_i log2(e),
// or -inf where LSE_i = -inf; rows in [Nq, nq_pad) get nd = 0, nlse2 = -inf.
// d/8 lanes per row, one 16-byte load of O and of dO each.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdPreParams p) {
  constexpr int kLanes = D / 8;
  const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = g / kLanes;
  const int part = static_cast<int>(g % kLanes);
  const long long rows = static_cast<long long>(p.BH) * p.nq_pad;
  const bool live = row < rows;
  const long long bh = live ? row / p.nq_pad : 0;
  const int r = live ? static_cast<int>(row % p.nq_pad) : 0;
  float acc = 0.f;
  if (live && r < p.Nq) {
    const size_t e = (static_cast<size_t>(bh) * p.Nq + r) * D + part * 8;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + e));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + e));
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(wa[k] << 16), __uint_as_float(wb[k] << 16), acc);
      acc = fmaf(__uint_as_float(wa[k] & 0xFFFF0000u), __uint_as_float(wb[k] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o, kLanes);
  if (live && part == 0) {
    float nl2 = -INFINITY;
    if (r < p.Nq) {
      const float lse = p.lse[static_cast<size_t>(bh) * p.Nq + r];
      nl2 = lse == -INFINITY ? -INFINITY : -(lse * 1.4426950408889634f);
    } else {
      acc = 0.f;
    }
    p.nlse2[row] = nl2;
    p.nd[row] = -acc;
  }
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap* maps, const BwdParams& p, const BwdPreParams& pre,
                         cudaStream_t s) {
  using C = BwdCfg<D>;
  {
    const long long threads = static_cast<long long>(pre.BH) * pre.nq_pad * (D / 8);
    fa_bwd_pre_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(pre);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // maps: q, k, v, dout, dq, dk, dv
  auto ka = fa_bwd_dkdv_kernel<D>;
  // The setmaxnreg split assumes exactly kRegLaunchA registers per thread at launch.
  static const bool regs_ok = [&] {
    cudaFuncAttributes attr{};
    return cudaFuncGetAttributes(&attr, ka) == cudaSuccess && attr.numRegs == C::kRegLaunchA;
  }();
  if (!regs_ok) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemA);
  if (e != cudaSuccess) return e;
  const dim3 grid_a((p.Nk + C::kRows - 1) / C::kRows, p.BH);
  ka<<<grid_a, C::kThreads, C::kSmemA, s>>>(maps[0], maps[3], maps[1], maps[2], maps[5], maps[6], p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto kb = fa_bwd_dq_kernel<D>;
  e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemB);
  if (e != cudaSuccess) return e;
  const dim3 grid_b((p.Nq + C::kRows - 1) / C::kRows, p.BH);
  kb<<<grid_b, C::kThreads, C::kSmemB, s>>>(maps[0], maps[3], maps[1], maps[2], maps[4], p);
  return cudaGetLastError();
}

}  // namespace fa
