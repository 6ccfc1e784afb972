// fa_fwd_kernel.cuh -- single-pass tiled attention forward with the online
// softmax recurrence, for sm_103a (tcgen05 + TMEM + TMA + mbarrier).
//
// What it computes, per query row i of head (b, h):
//   for each K/V tile j:  S = Q K_j^T                      (tcgen05.mma, TMEM)
//                         m' = max(m, rowmax S)
//                         alpha = exp(m - m'); l <- alpha l; O <- alpha O
//                         P = exp(S - m'); l <- l + rowsum P; O <- O + P V_j
//   O <- O / l once at the end, LSE = scale * m + ln l.
// (Recurrence: "Online Softmax 算法详解" sections 2.3 and 3.2, "在线Softmax算法解析"
// section 3.2, "La recurrencia del online softmax" section "La recurrencia".)
// The scale is folded into a base-2 exponent, exp(scale*(s - m)) =
// 2^(s*c - m*c) with c = scale*log2(e): one FFMA + one EX2 per score
// ("Online Softmax 算法详解" section 5).  A row whose running max is still -inf
// uses 0 as its reference point, so no (-inf) - (-inf) appears (section 7.1);
// a row with l = 0 gets O = 0 and LSE = -inf (sections 7.2-7.3).
//
// CTA = QT query tiles of 128 rows of one (b, h), over one range of K/V tiles
// (the whole key axis, or one split of it).  The mask keeps, for query row r,
// keys [r + off - wl, r + off + wr] (off = Nk - Nq, -1 = open side; causal is
// (-1, 0)).  The CTA streams the K/V tiles from the first one any of its rows
// can see; every query tile starts there and stops after its own last visible
// tile, so the query tiles' ranges are prefixes of one stream.
//   WG 0          warp 0: TMA producer (one thread): Q once, then K and V
//                 tiles through a ring of shared-memory stages, K one step
//                 ahead of V (see ring_pos_k / ring_pos_v).
//                 Warp 1 + i: MMA issuer of tile i (warp-uniform code, one
//                 elected lane issues, blocking barrier waits):
//                 S_i(j+1) = Q_i K_{j+1}^T into its S buffer as soon as that
//                 is free (so it overlaps this tile's exponentials), then
//                 O_i += P_i(j) V_j (A = P_i from TMEM) once P_i(j) and the O
//                 rescale are in place.  Warp 3 allocates TMEM.
//   WG 1 + i      tile i.  Thread t owns row t of the tile (TMEM lane t), so
//                 row max and row sum are register-local (no shuffles).  Each
//                 step: read S_i, write P_i (bf16 pairs or E4M3 quads) to
//                 TMEM; bf16 rows seldom move their reference, and the warp
//                 rescales its own rows of O when one does.  Also runs the
//                 epilogue of its tile.
//   WG 1 + QT     E4M3 only -- correction: rows follow the exact max and
//                 rescale on most steps, so O_i <- alpha O_i runs here, beside
//                 the softmax, once P_i(j-1).V_{j-1} has landed; a warp whose
//                 32 rows all keep their max releases the step at once.
// setmaxnreg moves registers from the producer (and correction) warpgroups to
// the softmax warpgroups.
// TMEM (32-bit columns): S_i (BC columns per tile where 512 columns hold
// everything, else one S buffer that the tiles take in turn: S_0(0), S_1(0),
// S_0(1), ...), P_i (BC/2 or BC/4 columns), O_i (D columns each).  P_i(j+1)
// is written only after O_i += P_i(j) V_j has completed.  Shared memory: the
// Q tiles ([128 rows][D], 128-byte swizzle, the layout the MMA reads K-major),
// then the K/V ring: keeping P out of shared memory leaves room for five 32 KB
// stages at d = 128.
// Softmax reference: bf16 rows move their reference m only when the tile max
// exceeds it by more than 16 in base-2 exponent units (P <= 2^16), so O is
// rarely rescaled; the final O / l and LSE do not depend on the reference.
//
// Every mbarrier wait is bounded by a global-timer limit.  A wait that runs
// out sets the CTA's abort flag and the device status word; every role then
// leaves its loop, lets its own copies / MMAs in flight finish, and the CTA
// frees TMEM and exits without writing outputs.
#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_wait.cuh"

namespace fa {

// F8: Q, K, V and P are FP8 E4M3 (one byte per element) and the products use
// tcgen05.mma kind::f8f6f4; everything else -- roles, ring, recurrence -- is
// shared with the bf16 kernel.
template <int D, int BC, int QT, bool F8 = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!F8 || (D == 128 && BC == 128), "FP8: d = 128, 128-key tiles");
  static constexpr int kEs = F8 ? 1 : 2;           // bytes per Q / K / V / P element
  static constexpr int kChunkElems = 128 / kEs;    // elements per 128-byte swizzle row
  static constexpr int kKStep = 32 / kEs;          // elements per MMA K-step (32 bytes)
  static_assert(BC == 64 || BC == 128, "K/V tile");
  static_assert(QT == 1 || QT == 2, "Q tiles per CTA");
  static constexpr int kBr = 128;  // query rows per tile (= TMEM lanes)
  // A separate correction warpgroup rescales O for E4M3, whose rows move
  // their max (and so rescale) on most steps.  bf16 rows rarely rescale (see
  // kLazy); their softmax warpgroup does it itself.
  static constexpr bool kCorr = F8;
  static constexpr int kWGs = QT + (kCorr ? 2 : 1);
  // Warpgroup 0 holds the producer, MMA and TMEM-allocation warps; softmax
  // tile i is warpgroup 1 + i, the E4M3 correction warpgroup comes last.
  static constexpr int kCorrWG = kCorr ? QT + 1 : -1;  // correction warpgroup
  static constexpr int kLoadWarp = 0;
  static constexpr int kMmaWarp0 = kLoadWarp + 1;  // + i: issuer of tile i
  static constexpr int kAllocWarp = kLoadWarp + 3;
  static constexpr int kThreads = 128 * kWGs;
  // Registers per thread at launch (65536 / threads, multiple of 8) and the
  // setmaxnreg split that moves them to the softmax warpgroups.  The split must
  // add up to what the block launches with, or setmaxnreg.inc would wait forever.
  // 256 threads launch with the per-thread maximum and need no split.
  static constexpr bool kSplitRegs = kThreads > 256;
  static constexpr int kRegLaunch = kCorr ? (QT == 2 ? 128 : 168) : (QT == 2 ? 168 : 0);
  static constexpr int kRegSoftmax = kCorr ? (QT == 2 ? 192 : 216) : (QT == 2 ? 216 : 0);
  static constexpr int kRegCorr = kCorr ? (QT == 2 ? 64 : 160) : 0;
  static constexpr int kRegOther = kCorr ? (QT == 2 ? 64 : 128) : (QT == 2 ? 72 : 0);
  static_assert(!kSplitRegs || QT * kRegSoftmax + kRegCorr + kRegOther == kWGs * kRegLaunch,
                "setmaxnreg split must add up to the registers the block launches with");
  static_assert(kRegLaunch * kThreads <= 65536, "launch register budget");
  static constexpr int kChunks = D / kChunkElems;  // 128-byte swizzle chunks per row
  static constexpr int kQChunkBytes = kBr * 128;  // 128 rows x 128 B
  static constexpr int kQTileBytes = kChunks * kQChunkBytes;
  static constexpr int kPCols = BC * kEs / 4;  // TMEM columns of P_i (packed pairs / quads)
  // Growth of the row max (base-2 exponent units) absorbed without moving the
  // softmax reference: bf16 P up to 2^16 (O and l stay far inside fp32 for
  // any key count); E4M3 P' already spans its range.
  static constexpr float kLazy = F8 ? 0.f : 16.f;
  static constexpr int kKVChunkBytes = BC * 128;
  static constexpr int kKVTileBytes = kChunks * kKVChunkBytes;
  // TMEM (32-bit columns): S, P_i, then O_i (starting on a multiple of D).
  // Each tile has its own S buffer where that fits in 512 columns; otherwise
  // one S buffer that the tiles take in turn.
  static constexpr bool kSharedS = QT * (BC + kPCols + D) > 512;
  static constexpr int kSBufs = kSharedS ? 1 : QT;
  static constexpr int kSCol = 0;
  static constexpr int kPCol = kSBufs * BC;
  static constexpr int kOCol = (kPCol + QT * kPCols + D - 1) / D * D;
  static constexpr int kTmemNeed = kOCol + QT * D;
  static constexpr int kTmemCols = kTmemNeed <= 64    ? 64
                                   : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256
                                                      : 512;
  static constexpr int kCtlBytes = 2048;
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int kStagesFit =
      (kSmemLimit - 1024 - kCtlBytes - QT * kQTileBytes) / kKVTileBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static_assert(kStages >= 2, "shared memory");
  static constexpr int kSmemBytes =
      1024 + QT * kQTileBytes + kStages * kKVTileBytes + kCtlBytes;
};

struct __align__(8) Ctl {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8][2];  // [stage][tile]: that tile's MMAs reading the stage completed
  uint64_t s_full[2];       // S_i(j) in TMEM (MMA commit)
  uint64_t s_free[2];       // all 128 rows of S_i(j) read into registers (128 arrivals)
  uint64_t alpha_full[2];   // alpha_i(j) published (128 softmax arrivals)
  uint64_t alpha_free[2];   // alpha_i(j) read by the correction (128 arrivals)
  uint64_t pv_ready[2];     // P_i(j) in TMEM and O_i rescaled (128 softmax [+ 128 correction] arrivals)
  uint64_t o_done[2];       // O_i += P_i(j) V_j completed (MMA commit)
  uint64_t drain[2];        // every MMA of tile i's issuer has completed
  uint32_t tmem_base;
  int abort;
  float alpha[2][128];      // per-row rescale factor, softmax -> correction
};
static_assert(sizeof(Ctl) <= 2048, "control block");

// Order of the K/V tiles through the shared-memory ring for a CTA with n steps:
// K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}: K runs one step
// ahead of V, as S_i(j+1) is computed while step j's softmax still runs.
__device__ __forceinline__ int ring_pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int ring_pos_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }
// Inverse: position p -> (is_v, step).
__device__ __forceinline__ void ring_decode(int p, int n, bool& is_v, int& step) {
  if (p == 0) {
    is_v = false, step = 0;
  } else if (p == 2 * n - 1) {
    is_v = true, step = n - 1;
  } else if (p & 1) {
    is_v = false, step = (p + 1) >> 1;
  } else {
    is_v = true, step = (p - 2) >> 1;
  }
}

template <int D, int BC, int QT, bool F8 = false>
__global__ void __launch_bounds__(FwdCfg<D, BC, QT, F8>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using C = FwdCfg<D, BC, QT, F8>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the shared-space address (128-byte swizzle atoms).
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + QT * C::kQTileBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(sKV + C::kStages * C::kKVTileBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work coordinates (identical in every thread)
  const int qg = p.causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  const int split = blockIdx.y;
  const int bh = blockIdx.z;
  const int row0 = qg * (C::kBr * QT);
  const int kv_begin = split * p.tiles_per_split;
  const int kv_end = min(p.kv_tiles, kv_begin + p.tiles_per_split);
  // K/V tiles [b_i, e_i) of this split hold keys visible to rows of query
  // tile i (empty: e_i = b_i).  The CTA streams from cta_b = min b_i; tile i
  // takes steps [0, n_i) of that stream, n_i = e_i - cta_b (its leading tiles
  // before b_i are fully masked for it and cost one MMA pair each).
  const int off = p.Nk - p.Nq;
  int n_i[QT];
  int cta_b = kv_end, kv_end_cta = kv_begin;
  bool any_tile = false;  // a split past the last K/V tile has kv_begin >= kv_end
#pragma unroll
  for (int i = 0; i < QT; ++i) {
    const int r_first = row0 + C::kBr * i;
    n_i[i] = -1;  // end tile, -1 = none
    if (r_first < p.Nq) {
      const int r_last = min(r_first + C::kBr, p.Nq) - 1;
      // |r + off| < 2^30 and wl, wr <= 2^30: these sums stay within int
      const int klo = p.wl < 0 ? 0 : max(0, r_first + off - p.wl);
      const int khi = p.wr < 0 ? p.Nk - 1 : min(p.Nk - 1, r_last + off + p.wr);
      if (khi >= klo) {
        const int b = max(kv_begin, static_cast<int>(klo / BC));
        const int e = min(kv_end, static_cast<int>(khi / BC) + 1);
        if (e > b) {
          n_i[i] = e;
          any_tile = true;
          cta_b = min(cta_b, b);
          kv_end_cta = max(kv_end_cta, e);
        }
      }
    }
  }
  if (!any_tile) cta_b = kv_end_cta = kv_begin;  // nothing to stream
#pragma unroll
  for (int i = 0; i < QT; ++i) n_i[i] = n_i[i] < 0 ? 0 : n_i[i] - cta_b;

  const uint32_t bar_q = smem_u32(&ctl->q_full);
  const uint32_t bar_kv_full = smem_u32(&ctl->kv_full[0]);
  const uint32_t bar_kv_empty = smem_u32(&ctl->kv_empty[0][0]);  // + 16*stage + 8*tile
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_sfree = smem_u32(&ctl->s_free[0]);
  const uint32_t bar_alpha = smem_u32(&ctl->alpha_full[0]);
  const uint32_t bar_afree = smem_u32(&ctl->alpha_free[0]);
  const uint32_t bar_pv = smem_u32(&ctl->pv_ready[0]);
  const uint32_t bar_o = smem_u32(&ctl->o_done[0]);
  const uint32_t bar_drain = smem_u32(&ctl->drain[0]);

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full + 8 * s, 1);
      for (int i = 0; i < QT; ++i) mbar_init(bar_kv_empty + 16 * s + 8 * i, 1);
    }
    for (int i = 0; i < QT; ++i) {
      mbar_init(bar_s + 8 * i, 1);
      mbar_init(bar_sfree + 8 * i, 128);
      mbar_init(bar_alpha + 8 * i, 128);
      mbar_init(bar_afree + 8 * i, 128);
      mbar_init(bar_pv + 8 * i, C::kCorr ? 256 : 128);
      mbar_init(bar_o + 8 * i, 1);
      mbar_init(bar_drain + 8 * i, 1);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
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
  const int wg = warp >> 2;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes

  if (wg == 0) {
    if constexpr (C::kSplitRegs) setmaxnreg_dec<C::kRegOther>();
    if (warp == C::kLoadWarp) {
      if (lane == 0) {
      // ============================================================== producer
      uint32_t qbytes = 0;
#pragma unroll
      for (int i = 0; i < QT; ++i)
        if (n_i[i] > 0) qbytes += C::kQTileBytes;
      if (qbytes) {
        mbar_arrive_expect_tx(bar_q, qbytes);
#pragma unroll
        for (int i = 0; i < QT; ++i) {
          if (n_i[i] <= 0) continue;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem_u32(sQ + i * C::kQTileBytes + c * C::kQChunkBytes), &tm_q, bar_q,
                        c * C::kChunkElems, row0 + C::kBr * i, bh);
        }
      }
      uint32_t issued_mask = 0, issued_par = 0;
      const int n_cta = kv_end_cta - cta_b;
      bool ok = true;
      for (int it = 0; ok && it < 2 * n_cta; ++it) {
        const int stage = it % C::kStages;
        const int use = it / C::kStages;
        if (use > 0) {
          // the slot's previous content (ring position it - kStages) must be
          // released by every tile that read it
          bool pv_;
          int prev_step;
          ring_decode(it - C::kStages, n_cta, pv_, prev_step);
#pragma unroll
          for (int i = 0; i < QT; ++i)
            if (ok && prev_step < n_i[i])
              ok = wait_bounded(bar_kv_empty + 16 * stage + 8 * i, (use - 1) & 1, wc);
          if (!ok) break;
        }
        if (it == p.test_skip_load) continue;  // test hook: this slot never fills
        bool is_v;
        int step;
        ring_decode(it, n_cta, is_v, step);
        const uint32_t full = bar_kv_full + 8 * stage;
        mbar_arrive_expect_tx(full, C::kKVTileBytes);
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem_u32(sKV + stage * C::kKVTileBytes + c * C::kKVChunkBytes), map, full,
                      c * C::kChunkElems, (cta_b + step) * BC, bh);
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (static_cast<uint32_t>(use & 1) << stage);
      }
      // Every copy started here must land before the CTA may exit.
      for (int s = 0; s < C::kStages; ++s)
        if ((issued_mask >> s) & 1u) wait_own(bar_kv_full + 8 * s, (issued_par >> s) & 1u, p.timeout_ns);
      if (qbytes) wait_own(bar_q, 0, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp >= C::kMmaWarp0 && warp < C::kMmaWarp0 + QT) {
      // ====================================================== MMA issuer, tile i
      const int i = warp - C::kMmaWarp0;
      // K-major A (Q), B (K); PV: A = P K-major, B = V MN-major
      constexpr uint32_t kIdescQK = F8 ? idesc_e4m3_f32(128, BC, false) : idesc_bf16_f32(128, BC, false);
      constexpr uint32_t kIdescPV = F8 ? idesc_e4m3_f32(128, D, true) : idesc_bf16_f32(128, D, true);
      auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
        if constexpr (F8)
          mma_e4m3_ss_elect(d, a, b, idesc, acc);
        else
          mma_bf16_ss_elect(d, a, b, idesc, acc);
      };
      auto mma_ts = [&](uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
        if constexpr (F8)
          mma_e4m3_ts_elect(d, a_tmem, b, idesc, acc);
        else
          mma_bf16_ts_elect(d, a_tmem, b, idesc, acc);
      };
      // Descriptor templates; the start-address field (bits 0-13, address >> 4)
      // of a shared address below 256 KB never carries, so per-MMA offsets are
      // plain 32-bit adds to the low word.
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ + i * C::kQTileBytes), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sKV), C::kKVChunkBytes, 1024);
      const uint64_t hi_q = dq0 & 0xFFFFFFFF00000000ull, hi_k = dk0 & 0xFFFFFFFF00000000ull,
                     hi_v = dv0 & 0xFFFFFFFF00000000ull;
      const uint32_t lo_q = static_cast<uint32_t>(dq0), lo_k = static_cast<uint32_t>(dk0),
                     lo_v = static_cast<uint32_t>(dv0);
      const uint32_t tS = tmem + C::kSCol + (C::kSharedS ? 0 : i * BC),
                     tP = tmem + C::kPCol + i * C::kPCols,
                     tO = tmem + C::kOCol + i * D;
      const int n = n_i[i];
      const int n_cta = kv_end_cta - cta_b;
      auto kv_ready = [&](int pos) {
        return warp_wait(bar_kv_full + 8 * (pos % C::kStages), (pos / C::kStages) & 1, wc);
      };
      // A shared S buffer is taken in the order S_0(0), S_1(0), S_0(1), ...
      // (a tile past its last step drops out); a tile's own buffer holds
      // S_i(0), S_i(1), ...  Each use waits until the previous one has been
      // read into registers.  Previous use before S_i(q): bar / parity of its
      // s_free, false if none.
      auto prev_use = [&](int q, uint32_t& bar, uint32_t& par) {
        if constexpr (QT == 2 && C::kSharedS) {
          const int o = 1 - i, qo = i == 1 ? q : q - 1;
          if (qo >= 0 && qo < n_i[o]) {
            bar = bar_sfree + 8 * o, par = qo & 1;
            return true;
          }
        }
        if (q == 0) return false;
        bar = bar_sfree + 8 * i, par = (q - 1) & 1;
        return true;
      };
      auto s_ready = [&](int q) {  // S_i(q) may be written: the buffer's previous product was read
        uint32_t bar, par;
        return !prev_use(q, bar, par) || warp_wait(bar, par, wc);
      };
      auto issue_qk = [&](int q) {  // S_i(q) = Q_i K_q^T, then release K_q's slot for tile i
        const int stage = ring_pos_k(q) % C::kStages;
        const uint32_t k_lo = lo_k + ((stage * C::kKVTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / C::kKStep; ++kk) {  // 32 bytes of K per step
          const uint32_t off_q = ((kk / 4) * C::kQChunkBytes + (kk % 4) * 32) >> 4;
          const uint32_t off_k = ((kk / 4) * C::kKVChunkBytes + (kk % 4) * 32) >> 4;
          mma(tS, hi_q | (lo_q + off_q), hi_k | (k_lo + off_k), kIdescQK, kk > 0);
        }
        mma_commit_elect(bar_s + 8 * i);
        mma_commit_elect(bar_kv_empty + 16 * stage + 8 * i);
      };
      auto issue_pv = [&](int v) {  // O_i += P_i(v) V_v, then release V_v's slot for tile i
        const int stage = ring_pos_v(v, n_cta) % C::kStages;
        const uint32_t v_lo = lo_v + ((stage * C::kKVTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < BC / C::kKStep; ++kk) {
          // P: one K-step (32 bytes = 8 TMEM columns of packed P).  V: kKStep
          // keys = 8-row groups of 1024 B (SBO); D columns in 128-byte chunks
          // BC*128 B apart (LBO).
          mma_ts(tO, tP + 8 * kk, hi_v | (v_lo + ((kk * C::kKStep * 128) >> 4)), kIdescPV,
                 (v > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit_elect(bar_o + 8 * i);
        mma_commit_elect(bar_kv_empty + 16 * stage + 8 * i);
      };
      // S_i(j+1) first: it waits only for the other tile to read its S, which
      // comes before P_i(j) is ready.
      bool ok = n > 0;
      bool issued = false;
      if (ok) ok = warp_wait(bar_q, 0, wc) && s_ready(0) && kv_ready(ring_pos_k(0));
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        issued = true;
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          ok = s_ready(j + 1) && kv_ready(ring_pos_k(j + 1));
          if (!ok) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        // O_i += P_i(j) V_j once P_i(j) is in TMEM and O_i rescaled
        ok = warp_wait(bar_pv + 8 * i, j & 1, wc) && kv_ready(ring_pos_v(j, n_cta));
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
      }
      if (issued) {
        // Everything issued above completes before TMEM may be freed.
        mma_commit_elect(bar_drain + 8 * i);
        wait_own(bar_drain + 8 * i, 0, p.timeout_ns);
      }
      __syncwarp();
    }
  } else if (C::kCorr && wg == C::kCorrWG) {
    // ========================================================= correction
    // Serves the tiles in whatever order their inputs arrive: per tile,
    // (1) read alpha_i(j) as soon as it is published and release the slot,
    // (2) once O_i += P_i(j-1) V_{j-1} has completed, O_i <- alpha O_i, then
    // let the MMA warp issue O_i += P_i(j) V_j.
    if constexpr (C::kSplitRegs && C::kRegCorr < C::kRegLaunch) setmaxnreg_dec<C::kRegCorr>();
    const int t = threadIdx.x & 127;
    int jn[QT];        // next step of tile i
    bool have[QT];     // alpha_i(jn) read, waiting for the previous P.V
    float alpha_r[QT];
#pragma unroll
    for (int i = 0; i < QT; ++i) {
      jn[i] = 0;
      have[i] = false;
      alpha_r[i] = 1.f;
    }
    auto probe = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_test(bar, parity));
    };
    uint32_t idle = 0;
    uint64_t t_idle = 0;
    bool ok = true;
    while (ok) {
      bool done = true, progressed = false;
#pragma unroll
      for (int i = 0; i < QT; ++i) {
        const int j = jn[i];
        if (j >= n_i[i]) continue;
        done = false;
        if (!have[i]) {
          if (!probe(bar_alpha + 8 * i, j & 1)) {
            continue;
          }
          alpha_r[i] = ctl->alpha[i][t];
          mbar_arrive(bar_afree + 8 * i);  // the softmax may publish alpha_i(j+1)
          have[i] = true;
          progressed = true;
        }
        // A warp whose 32 rows all keep their reference (alpha = 1) has
        // nothing to rescale and releases the product at once.
        const float alpha = alpha_r[i];
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!probe(bar_o + 8 * i, (j - 1) & 1)) {
            continue;
          }
          {
            tc_fence_after();
            const uint32_t tO = tmem + lane_off + C::kOCol + i * D;
            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
              uint32_t o[32];
              tmem_ld32_sync(tO + cc, o);
#pragma unroll
              for (int k = 0; k < 32; k += 2) {
                float y0, y1;
                f2_unpack(fmul2(f2_pack(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), a2), y0, y1);
                o[k] = __float_as_uint(y0);
                o[k + 1] = __float_as_uint(y1);
              }
              tmem_st32(tO + cc, o);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(bar_pv + 8 * i);
        have[i] = false;
        jn[i] = j + 1;
        progressed = true;
      }
      if (done) break;
      if (progressed) {
        idle = 0;
        continue;
      }
      // Nothing ready: poll again (a suspended wait on one tile's input
      // reacts late to the other tile's).
      if ((idle++ & 63) == 0) {
        const uint64_t now = global_timer_ns();
        if (idle == 1) t_idle = now;
        if (__any_sync(0xffffffffu, *wc.abort != 0)) break;
        if (now - t_idle > p.timeout_ns) {
          if ((threadIdx.x & 31) == 0) {
            *wc.abort = 1;
            atomicExch(p.status, kDevTimeout);
          }
          break;
        }
      }
    }
  } else {
    // ========================================================== tile i
    if constexpr (C::kSplitRegs) setmaxnreg_inc<C::kRegSoftmax>();
    const int i = wg - 1;
    const int t = threadIdx.x & 127;
    const uint32_t tS = tmem + lane_off + C::kSCol + (C::kSharedS ? 0 : i * BC);
    const uint32_t tP = tmem + lane_off + C::kPCol + i * C::kPCols;
    const uint32_t tO = tmem + lane_off + C::kOCol + i * D;
    const int row = row0 + C::kBr * i + t;
    const int n = n_i[i];
    const float c = p.scale_log2;
    // The row sits at key position rq = row + Nk - Nq; keys visible to it are
    // [rq - wl, rq + wr] within [0, Nk), a -1 bound leaving that side open.
    // (|rq| < 2^30 and wl, wr <= 2^30, so the sums below stay within int.)
    // K/V tiles [jf_b, jf_e) hold only keys that every row of this query tile
    // sees; they skip the mask (a test uniform across the warpgroup).
    const int rq = row + off;
    int jf_b = 0, jf_e;
    {
      const int tr_first = row0 + C::kBr * i + off;
      const int tr_last = min(row0 + C::kBr * (i + 1), p.Nq) - 1 + off;
      if (p.wl >= 0) {
        const int lo = tr_last - p.wl;  // highest first-visible key of the tile's rows
        jf_b = lo <= 0 ? 0 : (lo + BC - 1) / BC;
      }
      const int hi = p.wr < 0 ? p.Nk - 1 : min(p.Nk - 1, tr_first + p.wr);  // lowest last-visible key
      jf_e = hi < 0 ? 0 : (hi + 1) / BC;
    }

    bool ok = true;
    float m = -INFINITY;
    float l = 0.f;
    // bf16: sum over the tiles of bf16(P) - P at each tile's max element,
    // rescaled like l.  O is normalised by l + l_fix, so the largest weights
    // of a row enter O and its normaliser with the same rounding; LSE uses l.
    float l_fix = 0.f;
    for (int jj = 0; ok && jj < n; ++jj) {
      const int j = cta_b + jj;
      if (!warp_wait(bar_s + 8 * i, jj & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();

      uint32_t r[BC];
      if constexpr (BC == 128)
        tmem_ld64x2_sync(tS, tS + 64, r);
      else
        tmem_ld64_sync(tS, r);
      tc_fence_before();
      mbar_arrive(bar_sfree + 8 * i);  // the S buffer may take the next product
      float s[BC];
#pragma unroll
      for (int cc = 0; cc < BC; ++cc) s[cc] = __uint_as_float(r[cc]);
      if (j < jf_b || j >= jf_e) {  // key-axis tail, causal diagonal, window edge
        const int key0 = j * BC;
        const int lim = p.wr < 0 ? p.Nk - 1 : min(p.Nk - 1, rq + p.wr);
        const int lim_lo = p.wl < 0 ? 0 : rq - p.wl;
#pragma unroll
        for (int cc = 0; cc < BC; ++cc)
          if (key0 + cc > lim || key0 + cc < lim_lo) s[cc] = -INFINITY;
      }

      // m' = max(m, rowmax S): four independent chains of three-input max
      float mx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
      for (int cc = 8; cc < BC; cc += 2) mx[(cc >> 1) & 3] = max3f(mx[(cc >> 1) & 3], s[cc], s[cc + 1]);
      // The reference m moves to the tile's max only when that lies more
      // than C::kLazy (base-2 exponent units) above it, so P stays within
      // [0, 2^kLazy] and most steps leave O alone (alpha = 1).  The final
      // O / l and LSE = m scale + ln l are the same for any reference.
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const bool bump = mt > m && (m == -INFINITY || (mt - m) * c > C::kLazy);
      const float m_new = bump ? mt : m;
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = bump ? ex2_approx((m - m_ref) * c) : 1.f;
      if constexpr (C::kCorr) {
        // The correction must have read alpha_i(j-1) before the slot is reused
        // (S_i(j) was issued before it ran, so this step can be ahead of it).
        if (jj > 0 && !warp_wait(bar_afree + 8 * i, (jj - 1) & 1, wc)) {
          ok = false;
          break;
        }
        ctl->alpha[i][t] = alpha;  // the correction warpgroup rescales O_i by it
        mbar_arrive(bar_alpha + 8 * i);
      }

      // P = 2^(s*c - m_ref*c) (packed FFMA, then EX2); rowsum of the fp32 P
      // (before the cast to bf16 / E4M3) in four packed partial sums.  FP8:
      // Max_offset = 8 ("Online Softmax 算法详解" section 6): P' = 2^8 P, in
      // [0, 256], to use the E4M3 range; the sum of P' is scaled back by 2^-8
      // at the end and O by final_scale.
      const uint64_t c2 = f2_pack(c, c);
      const float neg = -m_ref * c + (F8 ? 8.f : 0.f);
      const uint64_t neg2 = f2_pack(neg, neg);
      float dfix = 0.f;
      if constexpr (!F8) {
        // P at the tile's max element, as the loop below computes it, and its
        // bf16 rounding (0 for a fully masked tile: 2^-inf).
        const float pm = ex2_approx(fmaf(mt, c, neg));
        dfix = __uint_as_float(pack_bf16x2(0.f, pm) & 0xFFFF0000u) - pm;
      }
      uint64_t ls[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ls[u] = 0ull;
      uint32_t pk[BC / (4 / C::kEs)];  // bf16 pairs or E4M3 quads
#pragma unroll
      for (int cc = 0; cc < BC; cc += 4) {
        float x0, x1, x2, x3;
        f2_unpack(ffma2(f2_pack(s[cc], s[cc + 1]), c2, neg2), x0, x1);
        f2_unpack(ffma2(f2_pack(s[cc + 2], s[cc + 3]), c2, neg2), x2, x3);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2);
        const float p3 = ex2_approx(x3);
        ls[(cc >> 1) & 3] = fadd2(ls[(cc >> 1) & 3], f2_pack(p0, p1));
        ls[((cc >> 1) + 1) & 3] = fadd2(ls[((cc >> 1) + 1) & 3], f2_pack(p2, p3));
        if constexpr (F8) {
          pk[cc >> 2] = pack_e4m3x4(p0, p1, p2, p3);
        } else {
          pk[cc >> 1] = pack_bf16x2(p0, p1);
          pk[(cc >> 1) + 1] = pack_bf16x2(p2, p3);
        }
      }
      float lsum[4];
      f2_unpack(fadd2(ls[0], ls[1]), lsum[0], lsum[1]);
      f2_unpack(fadd2(ls[2], ls[3]), lsum[2], lsum[3]);
      const float rowsum = (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
      // P_i(j) -> TMEM, row t in lane t (the A operand of O_i += P_i(j) V_j),
      // once O_i += P_i(j-1) V_{j-1} has finished reading the columns.
      if (jj > 0 && !warp_wait(bar_o + 8 * i, (jj - 1) & 1, wc)) {
        ok = false;
        break;
      }
      if constexpr (!C::kCorr) {
        // O_i <- alpha O_i for this warp's 32 rows, now that O_i += P_i(j-1)
        // V_{j-1} has landed; rare, as the reference seldom moves.
        if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          tc_fence_after();
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld32_sync(tO + cc, o);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float y0, y1;
              f2_unpack(fmul2(f2_pack(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), a2), y0, y1);
              o[k] = __float_as_uint(y0);
              o[k + 1] = __float_as_uint(y1);
            }
            tmem_st32(tO + cc, o);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < C::kPCols; u += 32) tmem_st32(tP + u, pk + u);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_pv + 8 * i);
      l = alpha * l + rowsum;
      l_fix = alpha * l_fix + dfix;
      m = m_new;
    }
    if (ok && n > 0) ok = warp_wait(bar_o + 8 * i, (n - 1) & 1, wc);
    const bool bad = named_bar_or(1 + i, 128, !ok || *wc.abort);
    // A tile that starts past the last query row has nothing to write.
    if (!bad && row0 + C::kBr * i < p.Nq) {
      if (n > 0) tc_fence_after();
      const bool empty = !(l > 0.f);
      // FP8: sum_scale l <- l 2^-8 undoes Max_offset in the row sum, and
      // final_scale (p.o_scale = v_descale 2^-8) in O ("Online Softmax 算法详解"
      // section 6.3); both are powers of two or exact scalings.
      const float lc = F8 ? l * (1.f / 256.f) : l;
      const float inv = empty ? 0.f : (F8 ? p.o_scale / lc : 1.f / (l + l_fix));
      if (!p.partial) {
        // bf16 O, staged in this tile's (now unused) Q buffer with the 128-byte
        // swizzle, then TMA stores (rows past Nq are clipped by the map).  The
        // FP8 Q buffer holds one 64-column chunk of bf16 O at a time.
        const uint32_t stg = smem_u32(sQ + i * C::kQTileBytes);
        constexpr int kOChunks = D / 64;
        constexpr int kStageChunks = F8 ? 1 : kOChunks;  // O chunks staged per round
#pragma unroll
        for (int round = 0; round < kOChunks / kStageChunks; ++round) {
#pragma unroll
        for (int cc = round * 64 * kStageChunks; cc < (round + 1) * 64 * kStageChunks; cc += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32_sync(tO + cc, o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
          const int chunk = cc / 64 - round * kStageChunks;
          const int u0 = (cc % 64) / 8;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int u = u0 + q;
            st_shared_v4(stg + chunk * C::kQChunkBytes + t * 128 + ((u ^ (t & 7)) << 4), w[4 * q],
                         w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + i, 128);
        if (t == 0) {
#pragma unroll
          for (int ch = 0; ch < kStageChunks; ++ch)
            tma_store_3d(&tm_o, stg + ch * C::kQChunkBytes, (round * kStageChunks + ch) * 64,
                         row0 + C::kBr * i, bh);
          tma_store_commit();
          tma_store_wait_read();
        }
        if (kStageChunks < kOChunks) named_bar_sync(1 + i, 128);  // staging buffer free again
        }
        if (row < p.Nq)
          p.lse[static_cast<size_t>(bh) * p.Nq + row] = empty ? -INFINITY : m * p.scale + logf(lc);
      } else {
        // fp32 partial triple (m in natural-log units, l, O/l) for the merge.
        const size_t prow = (static_cast<size_t>(split) * p.BH + bh) * p.Nq + row;
        if (row < p.Nq) {
          p.m_part[prow] = empty ? -INFINITY : m * p.scale;
          p.l_part[prow] = empty ? 0.f : l;
        }
        float* op = p.o_part + prow * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32_sync(tO + cc, o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * inv);
          if (row < p.Nq) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_global_v4(op + cc + 4 * q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == C::kAllocWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int BC, int QT, bool F8 = false>
cudaError_t launch_fwd_t(const CUtensorMap* maps, const FwdParams& p, dim3 grid, cudaStream_t s) {
  using C = FwdCfg<D, BC, QT, F8>;
  auto kern = fa_fwd_kernel<D, BC, QT, F8>;
  // The setmaxnreg split assumes the block launches with exactly kRegLaunch
  // registers per thread; with fewer, setmaxnreg.inc could never be granted.
  static const bool regs_ok = [&] {
    cudaFuncAttributes attr{};
    return cudaFuncGetAttributes(&attr, kern) == cudaSuccess &&
           (!C::kSplitRegs || attr.numRegs == C::kRegLaunch);
  }();
  if (!regs_ok) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

}  // namespace fa
