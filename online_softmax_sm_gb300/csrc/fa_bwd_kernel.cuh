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
//     looping over the 128-query tiles that see it.  S^T = K_j Q^T (N = 128)
//     goes to a TMEM buffer that is free again as soon as the compute threads
//     have loaded it, so the next S^T overlaps this step's exponentials.
//     dP^T = V_j dO^T is issued per query half h (N = 64) into buffer h;
//     compute warpgroup h owns half h of every tile: thread t owns key t
//     (TMEM lane t), keeps P^T in registers, and writes P^T and dS^T (bf16
//     pairs) into the 64 buffer columns it has just read.  dV_j += P^T dO and
//     dK_j += dS^T Q take them as the TMEM A operand half by half, and each
//     half's buffer goes back to the next dP^T as soon as its dK is done, so
//     the two halves hand off independently.  Q_i sits in a ring one slot
//     deeper than dO_i's: it is read first (S^T) and released last (dK).
//   fa_bwd_dq_kernel  one 128-row query tile per CTA, Q_i and dO_i in shared
//     memory, looping over the key tiles it sees (K_j and V_j in rings of
//     their own: K_j is released by dQ, V_j already by dP): S = Q_i K_j^T and
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
#include "fa_status.h"
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
  // dK/dV kernel: Q_i in a ring of kQSlots, dO_i (with the row vectors
  // nlse2, nd) in a ring of kDoSlots.  A Q slot is needed first (S^T) and
  // released last (dK), so its ring is one slot deeper: Q_{i+1} lands while
  // step i - 1 still holds its slot.
  static constexpr int kQSlots = D == 128 ? 3 : 4;
  static constexpr int kDoSlots = D == 128 ? 2 : 4;
  static constexpr int kVecSlotBytes = 2 * kVecBytes;  // nlse2, nd
  // dQ kernel: K_j in a ring of kKSlots, V_j in a ring of kVSlots.  K_j is
  // read first (S) and released last (dQ), V_j only by dP, so the K ring is
  // the deeper one and a V load never waits for a dQ.
  static constexpr int kKSlots = D == 128 ? 3 : 4;
  static constexpr int kVSlots = D == 128 ? 2 : 4;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kCtlBytesA = 512;
  // K_j, V_j, the Q ring, the dO ring, the row vectors, the barriers.  At
  // d = 128 this leaves no room for padding: the dynamic shared memory base
  // must itself be 1024-byte aligned (checked at kernel entry).
  static constexpr int kSmemA = 2 * kTileBytes + kQSlots * kTileBytes + kDoSlots * kTileBytes +
                                kDoSlots * kVecSlotBytes + kCtlBytesA;
  static constexpr int kSmemB = 1024 + 2 * kTileBytes + (kKSlots + kVSlots) * kTileBytes + kCtlBytes;
  static_assert(kKSlots + kVSlots <= 8, "dQ kernel barriers");
  static_assert(kQSlots + kDoSlots <= 8, "dK/dV kernel barriers");
  static_assert(kSmemA <= 227 * 1024 && kSmemB <= 227 * 1024, "shared memory");
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
  // dK/dV kernel: S^T (fp32, 128 columns), the two dP^T half buffers (64
  // columns each, later P^T and dS^T pairs), then the two accumulators.
  static constexpr int kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
  // dQ kernel: S, dP, two bf16 dS buffers of 64 columns, dQ.
  static constexpr int kDPq = 128, kDS0 = 256, kDQ = 384;
};

struct __align__(8) BwdCtl {  // at most BwdCfg::kCtlBytesA bytes
  uint64_t fixed_full;  // K_j, V_j (dK/dV) or Q_i, dO_i (dQ) landed
  uint64_t full[8];     // ring stage / slot landed
  uint64_t empty[8];    // every MMA reading the stage / slot completed
  uint64_t s_full[2];   // S(^T) of this step in TMEM
  uint64_t s_free;      // S(^T) read by all 256 compute threads
  uint64_t dp_free;     // dQ kernel: dP read by all 256 compute threads
  uint64_t dp_full[2];  // dP(^T) in TMEM (dK/dV kernel: per query half)
  uint64_t ready[2];    // bf16 P^T (dK/dV kernel, per half) or dS (dQ kernel) written back to TMEM
  uint64_t ds_ready[2]; // dK/dV kernel: bf16 dS^T of a half written back to TMEM
  uint64_t done_b[2];   // dV and dK of a half done (its buffer free) / dQ MMA of a buffer done
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
  static_assert(sizeof(BwdCtl) <= C::kCtlBytesA, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  // The layout fills the shared memory limit, so it starts at the base
  // itself: a base that is not 1024-byte aligned (the 128-byte swizzle
  // atom) is reported and nothing runs.  The test is the same in every CTA.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kDevLayout);
    return;
  }
  uint8_t* sK = smem_raw;
  uint8_t* sV = sK + C::kTileBytes;
  uint8_t* sQr = sV + C::kTileBytes;                   // Q ring
  uint8_t* sDOr = sQr + C::kQSlots * C::kTileBytes;    // dO ring
  uint8_t* sVec = sDOr + C::kDoSlots * C::kTileBytes;  // per dO slot: nlse2[128], nd[128]
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sVec + C::kDoSlots * C::kVecSlotBytes);

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
  // Q slot i: full / empty[i]; dO slot j: full / empty[kQSlots + j]
  const uint32_t bar_qfull = smem_u32(&ctl->full[0]);
  const uint32_t bar_qempty = smem_u32(&ctl->empty[0]);
  const uint32_t bar_dofull = smem_u32(&ctl->full[C::kQSlots]);
  const uint32_t bar_doempty = smem_u32(&ctl->empty[C::kQSlots]);
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_sfree = smem_u32(&ctl->s_free);
  const uint32_t bar_dp = smem_u32(&ctl->dp_full[0]);
  const uint32_t bar_ready = smem_u32(&ctl->ready[0]);
  const uint32_t bar_dsr = smem_u32(&ctl->ds_ready[0]);
  const uint32_t bar_dk = smem_u32(&ctl->done_b[0]);
  const uint32_t bar_drain = smem_u32(&ctl->drain);

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kQSlots + C::kDoSlots; ++s) {
      mbar_init(bar_qfull + 8 * s, 1);
      mbar_init(bar_qempty + 8 * s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 256);  // every compute thread has its S^T columns in registers
    for (int h = 0; h < 2; ++h) {  // per query half h (dP^T buffer h, compute warpgroup h)
      mbar_init(bar_dp + 8 * h, 1);
      mbar_init(bar_ready + 8 * h, 128);  // the warpgroup's P^T pairs written
      mbar_init(bar_dsr + 8 * h, 128);    // and its dS^T pairs
      mbar_init(bar_dk + 8 * h, 1);       // dV and dK of the half done: buffer h free
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
      // per barrier (Q slots, then dO slots): a copy was issued; its parity
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      auto note = [&](int b, int use) {
        issued_mask |= 1u << b;
        issued_par = (issued_par & ~(1u << b)) | (static_cast<uint32_t>(use & 1) << b);
      };
      for (int s = 0; ok && s < n; ++s) {
        const int q0 = (i_lo + s) * C::kRows;
        // Q_s: its slot was last read by dK of step s - kQSlots
        const int qs = s % C::kQSlots, qu = s / C::kQSlots;
        if (qu > 0 && !wait_bounded(bar_qempty + 8 * qs, (qu - 1) & 1, wc)) {
          ok = false;
          break;
        }
        const uint32_t qfull = bar_qfull + 8 * qs;
        mbar_arrive_expect_tx(qfull, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sQr + qs * C::kTileBytes + c * C::kChunkBytes), &tm_q, qfull, c * 64, q0, bh);
        note(qs, qu);
        // dO_s, nlse2, nd: the slot was last read in step s - kDoSlots
        const int ds = s % C::kDoSlots, du = s / C::kDoSlots;
        if (du > 0 && !wait_bounded(bar_doempty + 8 * ds, (du - 1) & 1, wc)) {
          ok = false;
          break;
        }
        const uint32_t dfull = bar_dofull + 8 * ds;
        mbar_arrive_expect_tx(dfull, C::kTileBytes + 2 * C::kVecBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sDOr + ds * C::kTileBytes + c * C::kChunkBytes), &tm_do, dfull, c * 64, q0,
                      bh);
        const size_t vrow = static_cast<size_t>(bh) * p.nq_pad + q0;
        uint8_t* vec = sVec + ds * C::kVecSlotBytes;
        bulk_load(smem_u32(vec), p.nlse2 + vrow, C::kVecBytes, dfull, pol);
        bulk_load(smem_u32(vec + C::kVecBytes), p.nd + vrow, C::kVecBytes, dfull, pol);
        note(C::kQSlots + ds, du);
      }
      for (int b = 0; b < C::kQSlots + C::kDoSlots; ++b)
        if ((issued_mask >> b) & 1u) wait_own(bar_qfull + 8 * b, (issued_par >> b) & 1u, p.timeout_ns);
      if (n > 0) wait_own(bar_fixed, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp2) {
    // --------------------------------------------------------- MMA issuers
    // Query tile s (128 queries) per step.  S^T = K_j Q_s^T (N = 128) has a
    // TMEM buffer of its own, freed as soon as the compute threads have loaded
    // it into registers, so S^T(s+1) runs while P(s) is formed.  dP^T is
    // issued per query half h (N = 64) into buffer h, which compute
    // warpgroup h turns into bf16 pairs in place: P^T pairs in its first 32
    // columns, dS^T pairs in the next 32.  dV and dK then take the half's
    // four K-slices from TMEM, and dP^T(s+1, h) waits only for those, so the
    // two halves hand off independently.  Warp kMmaWarp2 issues S^T and dP^T,
    // warp kMmaWarp issues dV and dK.
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);  // A = K, B = Q (K-major)
    constexpr uint32_t kIdescDP = idesc_bf16_f32(128, 64, false);  // A = V, B = 64 rows of dO
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, true);   // B = dO or Q rows (MN-major)
    auto q_base = [&](int s) { return smem_u32(sQr + (s % C::kQSlots) * C::kTileBytes); };
    auto do_base = [&](int s) { return smem_u32(sDOr + (s % C::kDoSlots) * C::kTileBytes); };
    // TMEM column of the P^T pairs of K-slice kk (16 queries, 8 columns):
    // buffer kk / 4, 8 columns per slice; dS^T pairs 32 further
    auto a_col = [](int kk) { return static_cast<uint32_t>(C::kDP + 64 * (kk >> 2) + 8 * (kk & 3)); };
    bool ok = n > 0 && warp_wait(bar_fixed, 0, wc);
    if (warp == C::kMmaWarp2) {
      const uint64_t dK = desc_kmajor<D>(smem_u32(sK));
      const uint64_t dV = desc_kmajor<D>(smem_u32(sV));
      for (int s = 0; ok && s < n; ++s) {
        const uint32_t par = static_cast<uint32_t>((s - 1) & 1);
        ok = warp_wait(bar_qfull + 8 * (s % C::kQSlots), (s / C::kQSlots) & 1, wc) &&
             (s == 0 || warp_wait(bar_sfree, par, wc));
        if (!ok) break;
        tc_fence_after();
        const uint64_t dQk = desc_kmajor<D>(q_base(s));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // S^T = K_j Q_s^T
          mma_bf16_ss_elect(tmem + C::kS, dK + kslice_kmajor<D>(kk), dQk + kslice_kmajor<D>(kk), kIdescS,
                            kk > 0);
        mma_commit_elect(bar_s);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if ((s > 0 && !warp_wait(bar_dk + 8 * h, par, wc)) ||
              (h == 0 && !warp_wait(bar_dofull + 8 * (s % C::kDoSlots), (s / C::kDoSlots) & 1, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // rows [64 h, 64 h + 64) of dO_s: 64 rows of 128 bytes into each chunk
          const uint64_t dOk = desc_kmajor<D>(do_base(s) + 64 * 128 * h);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // dP^T (half h) = V_j dO_s,h^T
            mma_bf16_ss_elect(tmem + C::kDP + 64 * h, dV + kslice_kmajor<D>(kk), dOk + kslice_kmajor<D>(kk),
                              kIdescDP, kk > 0);
          mma_commit_elect(bar_dp + 8 * h);
        }
      }
    } else {
      for (int s = 0; ok && s < n; ++s) {
        const uint32_t par = static_cast<uint32_t>(s & 1);
        const uint64_t dOmn = desc_mnmajor<D>(do_base(s));
        const uint64_t dQmn = desc_mnmajor<D>(q_base(s));
        // half by half: dV once its P^T is written, dK once its dS^T is, then
        // the half's buffer goes back to dP^T(s+1, h) while the other half
        // is still being formed
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!warp_wait(bar_ready + 8 * h, par, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)  // dV += P^T dO_s (rows 16 kk)
            mma_bf16_ts_elect(tmem + C::kDV, tmem + a_col(kk), dOmn + kslice_mnmajor(kk), kIdescAcc,
                              (s > 0 || kk > 0) ? 1u : 0u);
          if (!warp_wait(bar_dsr + 8 * h, par, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)  // dK += dS^T Q_s
            mma_bf16_ts_elect(tmem + C::kDK, tmem + a_col(kk) + 32, dQmn + kslice_mnmajor(kk), kIdescAcc,
                              (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_elect(bar_dk + 8 * h);  // buffer h read by dV and dK
        }
        if (!ok) break;
        // S^T and dP^T of the step completed before P^T / dS^T were written
        // back, and the compute warps read nlse2 / nd before that: after dK
        // of both halves, nothing reads the step's Q or dO slot again
        mma_commit_elect(bar_qempty + 8 * (s % C::kQSlots));
        mma_commit_elect(bar_doempty + 8 * (s % C::kDoSlots));
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
    const int h = warp >> 2;               // query half of every tile
    const int t = (warp & 3) * 32 + lane;  // key row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int key = key0 + t;
    const float c = p.scale_log2;
    // this warpgroup's 64 columns of S^T and of dP^T
    const uint32_t tS = tmem + lane_off + C::kS + 64 * h;
    const uint32_t tDP = tmem + lane_off + C::kDP + 64 * h;
    bool ok = true;
    for (int s = 0; ok && s < n; ++s) {
      const int ds = s % C::kDoSlots;
      const int qt0 = (i_lo + s) * C::kRows;   // the tile's first query
      const int q0 = qt0 + 64 * h;             // this half's first query
      const float* nlv = reinterpret_cast<const float*>(sVec + ds * C::kVecSlotBytes) + 64 * h;
      const float* ndv = nlv + C::kRows;
      // The dO slot's barrier makes the bulk-copied nlse2 / nd visible here.
      ok = warp_wait(bar_dofull + 8 * ds, (s / C::kDoSlots) & 1, wc) && warp_wait(bar_s, s & 1, wc);
      if (!ok) break;
      tc_fence_after();
      const bool all_vis = bwd_tile_all_visible(qt0, key0, p);  // the whole 128 x 128 tile pair
      float pv[64];
      {
        uint32_t srow[64];
        tmem_ld64_sync(tS, srow);
        tc_fence_before();
        mbar_arrive(bar_sfree);  // S^T(s+1) may overwrite the buffer now
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
      // dP^T(s) of this half in buffer h: load it, then P^T pairs into the
      // first 32 of the columns just read (dV starts on them), then
      // dS^T = P^T (dP^T - D) into the next 32
      if (!warp_wait(bar_dp + 8 * h, s & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t drow[64];
      tmem_ld64_sync(tDP, drow);
      {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack_bf16x2(pv[2 * k], pv[2 * k + 1]);
        tmem_st32(tDP, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ready + 8 * h);
      {
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
        tmem_st32(tDP + 32, dk);
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
  uint8_t* sKr = sDO + C::kTileBytes;                // K ring
  uint8_t* sVr = sKr + C::kKSlots * C::kTileBytes;   // V ring
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(sVr + C::kVSlots * C::kTileBytes);

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
  // K slot i: full / empty[i]; V slot i: full / empty[kKSlots + i]
  const uint32_t bar_kfull = smem_u32(&ctl->full[0]);
  const uint32_t bar_kempty = smem_u32(&ctl->empty[0]);
  const uint32_t bar_vfull = smem_u32(&ctl->full[C::kKSlots]);
  const uint32_t bar_vempty = smem_u32(&ctl->empty[C::kKSlots]);
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_sfree = smem_u32(&ctl->s_free);
  const uint32_t bar_dp = smem_u32(&ctl->dp_full[0]);
  const uint32_t bar_dpfree = smem_u32(&ctl->dp_free);
  const uint32_t bar_ready = smem_u32(&ctl->ready[0]);    // + 8 b
  const uint32_t bar_dq = smem_u32(&ctl->done_b[0]);      // + 8 b
  const uint32_t bar_drain = smem_u32(&ctl->drain);

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kKSlots + C::kVSlots; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
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
      // per barrier (K slots, then V slots): a copy was issued; its parity
      uint32_t issued_mask = 0, issued_par = 0;
      for (int j = 0; j < n; ++j) {
        const int k0 = (j_lo + j) * C::kRows;
        const int ks = j % C::kKSlots, ku = j / C::kKSlots;  // K_j: slot last read by dQ(j - kKSlots)
        if (ku > 0 && !wait_bounded(bar_kempty + 8 * ks, (ku - 1) & 1, wc)) break;
        const uint32_t kfull = bar_kfull + 8 * ks;
        mbar_arrive_expect_tx(kfull, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sKr + ks * C::kTileBytes + c * C::kChunkBytes), &tm_k, kfull, c * 64, k0, bh);
        issued_mask |= 1u << ks;
        issued_par = (issued_par & ~(1u << ks)) | (static_cast<uint32_t>(ku & 1) << ks);
        const int vs = j % C::kVSlots, vu = j / C::kVSlots;  // V_j: slot last read by dP(j - kVSlots)
        if (vu > 0 && !wait_bounded(bar_vempty + 8 * vs, (vu - 1) & 1, wc)) break;
        const uint32_t vfull = bar_vfull + 8 * vs;
        mbar_arrive_expect_tx(vfull, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sVr + vs * C::kTileBytes + c * C::kChunkBytes), &tm_v, vfull, c * 64, k0, bh);
        const int vb = C::kKSlots + vs;
        issued_mask |= 1u << vb;
        issued_par = (issued_par & ~(1u << vb)) | (static_cast<uint32_t>(vu & 1) << vb);
      }
      for (int s = 0; s < C::kKSlots + C::kVSlots; ++s)
        if ((issued_mask >> s) & 1u) wait_own(bar_kfull + 8 * s, (issued_par >> s) & 1u, p.timeout_ns);
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
    auto k_slot = [&](int j) { return smem_u32(sKr + (j % C::kKSlots) * C::kTileBytes); };
    auto v_slot = [&](int j) { return smem_u32(sVr + (j % C::kVSlots) * C::kTileBytes); };
    bool ok = n > 0 && warp_wait(bar_fixed, 0, wc);
    if (warp == C::kMmaWarp) {
      const uint64_t dQk = desc_kmajor<D>(smem_u32(sQ));
      const uint64_t dOk = desc_kmajor<D>(smem_u32(sDO));
      for (int j = 0; ok && j < n; ++j) {
        ok = warp_wait(bar_kfull + 8 * (j % C::kKSlots), (j / C::kKSlots) & 1, wc) &&
             (j == 0 || warp_wait(bar_sfree, (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t dKk = desc_kmajor<D>(k_slot(j));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss_elect(tmem + C::kS, dQk + kslice_kmajor<D>(kk), dKk + kslice_kmajor<D>(kk),
                              kIdescS, kk > 0);
          mma_commit_elect(bar_s);
        }
        ok = warp_wait(bar_vfull + 8 * (j % C::kVSlots), (j / C::kVSlots) & 1, wc) &&
             (j == 0 || warp_wait(bar_dpfree, (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t dVk = desc_kmajor<D>(v_slot(j));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss_elect(tmem + C::kDPq, dOk + kslice_kmajor<D>(kk), dVk + kslice_kmajor<D>(kk),
                              kIdescS, kk > 0);
          mma_commit_elect(bar_dp);
          mma_commit_elect(bar_vempty + 8 * (j % C::kVSlots));  // V_j read
        }
      }
    } else {
      for (int j = 0; ok && j < n; ++j) {
        ok = warp_wait(bar_ready + 8 * (j & 1), (j >> 1) & 1, wc);  // dS(j) written back
        if (!ok) break;
        tc_fence_after();
        const uint64_t dKmn = desc_mnmajor<D>(k_slot(j));
        const uint32_t src = tmem + C::kDS0 + 64 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ += dS K_j (K = 128 keys, 8 columns per K-step)
          mma_bf16_ts_elect(tmem + C::kDQ, src + 8 * kk, dKmn + kslice_mnmajor(kk), kIdescDQ,
                            (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(bar_dq + 8 * (j & 1));
        // K_j: S(j) (the other warp) completed before dS(j) could exist
        mma_commit_elect(bar_kempty + 8 * (j % C::kKSlots));
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
