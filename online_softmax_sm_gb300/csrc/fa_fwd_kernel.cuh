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
// Persistent: the grid holds at most one CTA per SM, and each CTA walks a
// static list of work items.  An item is QT query tiles of 128 rows of one
// (b, h) over one range of K/V tiles (the whole key axis, or one split of
// it).  Items are dealt out in snake order (round r gives item r*G + c to CTA
// c on even rounds, r*G + G-1-c on odd ones), heaviest query tiles first when
// a mask makes their work unequal, so the CTAs' totals even out.  Everything
// that lives across items -- TMEM, the mbarriers and their phases, the K/V
// ring -- carries over: the next item's Q and first K/V tiles load while the
// current item finishes, and its first S product runs while the current
// epilogue drains.
//
// The mask keeps, for query row r, keys [r + off - wl, r + off + wr]
// (off = Nk - Nq, -1 = open side; causal is (-1, 0)).  An item streams the
// K/V tiles from the first one any of its rows can see; every query tile
// starts there and stops after its own last visible tile, so the query tiles'
// ranges are prefixes of one stream.
//   WG 0          warp 0: TMA producer (one thread): per item, Q_i, then K and
//                 V tiles through a ring of shared-memory stages, K one step
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
// a 16 KB O staging buffer per tile where it fits without dropping the K/V
// ring below five stages (else each tile's epilogue borrows a K/V ring slot
// for its O), then the K/V ring.
// Softmax reference: bf16 rows move their reference m only when the tile max
// exceeds it by more than 16 in base-2 exponent units (P <= 2^16), so O is
// rarely rescaled; the final O / l and LSE do not depend on the reference.
//
// Every mbarrier wait is bounded by a global-timer limit.  A wait that runs
// out sets the CTA's abort flag and the device status word; every role then
// leaves its loops, lets its own copies / MMAs in flight finish, and the CTA
// frees TMEM and exits without writing further outputs.
#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_wait.cuh"

#ifndef FA_STAGGER
#define FA_STAGGER 1
#endif

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
  static constexpr int kRegSoftmax = kCorr ? (QT == 2 ? 184 : 216) : (QT == 2 ? 216 : 0);
  static constexpr int kRegCorr = kCorr ? (QT == 2 ? 80 : 160) : 0;
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
  // Two tiles with S buffers of their own would run their softmax steps in
  // lockstep (both S products land together); tile 1 starts each item once
  // tile 0 has its first row maxima, so one tile's exponentials overlap the
  // other's loads and reductions.
  static constexpr bool kStagger = FA_STAGGER != 0 && QT == 2 && !kSharedS;
  static constexpr int kSBufs = kSharedS ? 1 : QT;
  static constexpr int kSCol = 0;
  static constexpr int kPCol = kSBufs * BC;
  static constexpr int kOCol = (kPCol + QT * kPCols + D - 1) / D * D;
  static constexpr int kTmemNeed = kOCol + QT * D;
  static_assert(kPCol >= kSCol + kSBufs * BC && kOCol >= kPCol + QT * kPCols, "TMEM regions overlap");
  static constexpr int kTmemCols = kTmemNeed <= 64    ? 64
                                   : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256
                                                      : 512;
  static_assert(kTmemNeed <= kTmemCols && kTmemCols <= 512, "TMEM columns");
  static constexpr int kCtlBytes = 2048;
  static constexpr int kSmemLimit = 227 * 1024;
  // bf16 O is staged for the TMA store 64 columns (one 128-byte swizzle row)
  // at a time: 16 KB per tile.
  static constexpr int kStgBytes = kBr * 128;
  static constexpr int kRingRoom = kSmemLimit - 1024 - kCtlBytes - QT * kQTileBytes;
  static constexpr int kStagesNoStg = kRingRoom / kKVTileBytes > 8 ? 8 : kRingRoom / kKVTileBytes;
  static constexpr int kStagesStg = (kRingRoom - QT * kStgBytes) / kKVTileBytes > 8
                                        ? 8
                                        : (kRingRoom - QT * kStgBytes) / kKVTileBytes;
  // O gets staging buffers of its own unless that costs a ring stage below
  // five; otherwise each item's epilogue borrows K/V ring slots (kSlotStg):
  // the producer hands out one slot per tile after the item's last K/V tile,
  // tile i stages all of its O in slot i, and the slot returns to the ring
  // once the store has read it.
  static constexpr bool kOwnStg = kStagesStg >= 5 || kStagesStg == kStagesNoStg;
  static constexpr bool kSlotStg = !kOwnStg;
  static constexpr int kStages = kOwnStg ? kStagesStg : kStagesNoStg;
  static_assert(kStages >= 2, "shared memory");
  static_assert(!kSlotStg || (kKVTileBytes >= D * 256 && kStages > QT), "O staging in ring slots");
  static constexpr int kSmemBytes =
      1024 + QT * kQTileBytes + (kOwnStg ? QT * kStgBytes : 0) + kStages * kKVTileBytes + kCtlBytes;
};

struct __align__(8) Ctl {
  uint64_t q_full[2];       // Q_i landed (TMA bytes)
  uint64_t q_free[2];       // Q_i buffer no longer read (last S_i product done; with O
                            // staged in it, the store has read it too)
  uint64_t kv_full[8];
  uint64_t kv_empty[8][2];  // [stage][tile]: that tile's MMAs reading the stage completed
  uint64_t s_full[2];       // S_i(j) in TMEM (MMA commit)
  uint64_t s_free[2];       // all 128 rows of S_i(j) read into registers (128 arrivals)
  uint64_t alpha_full[2];   // alpha_i(j) published (128 softmax arrivals)
  uint64_t alpha_free[2];   // alpha_i(j) read by the correction (128 arrivals)
  uint64_t pv_ready[2];     // P_i(j) in TMEM and O_i rescaled (128 softmax [+ 128 correction] arrivals)
  uint64_t o_done[2];       // O_i += P_i(j) V_j completed (MMA commit)
  uint64_t drain[2];        // every MMA of tile i's issuer has completed
  uint64_t stagger;         // tile 0 has its first row maxima of the item (kStagger)
  uint32_t tmem_base;
  int abort;
  int corr_stop[2];         // tile i has no more steps (E4M3 correction)
  float alpha[2][128];      // per-row rescale factor, softmax -> correction
};
static_assert(sizeof(Ctl) <= 2048, "control block");

// Order of the K/V tiles through the shared-memory ring for an item with n
// steps: K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}: K runs one
// step ahead of V, as S_i(j+1) is computed while step j's softmax still runs.
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

// Ring position -> (stage, phase parity): positions are counted from the
// start of the CTA; (base_stage, base_par) is the item's first position.
struct RingPos {
  int stage;
  uint32_t par;
};
template <int S>
__device__ __forceinline__ RingPos ring_at(int base_stage, uint32_t base_par, int p) {
  const int t = base_stage + p;
  return RingPos{t % S, base_par ^ (static_cast<uint32_t>(t / S) & 1u)};
}
template <int S>
__device__ __forceinline__ void ring_advance(int& base_stage, uint32_t& base_par, int n_pos) {
  const int t = base_stage + n_pos;
  base_stage = t % S;
  base_par ^= static_cast<uint32_t>(t / S) & 1u;
}

// One work item: query tiles [row0, row0 + 128 QT) of head bh over the K/V
// tiles of one split.  Tile i takes steps [0, n[i]) of the item's stream of
// n_cta K/V tiles starting at tile cta_b (n[i] = 0: no visible key).
template <int QT>
struct Item {
  int bh, split, row0;
  int cta_b, n_cta;
  int n[QT];
};

// Head, split and first query row of item `idx` (idx < n_items), in the
// order the host chose.
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  const unsigned int u = static_cast<unsigned int>(n);
  return static_cast<int>((__umulhi(u, f.mul) + u) >> f.shift);
}

template <int QT>
__device__ __forceinline__ void item_coords(int idx, const FwdParams& p, int& bh, int& split,
                                            int& row0) {
  int x;
  if (p.qg_major) {  // blocks of hb heads; in a block, query-tile group outermost (heaviest first)
    const int b = fdiv(idx, p.div_blk);
    const int rem = idx - b * p.div_blk.d;
    const FastDiv& per = (b + 1) * p.hb <= p.n_bh ? p.div_per : p.div_per_last;
    x = fdiv(rem, per);
    const int r = rem - x * per.d;
    const int hl = fdiv(r, p.div_split);
    bh = b * p.hb + hl;
    split = r - hl * p.n_split;
  } else {  // head outermost: the query tiles of one head are neighbours (L2 reuse of K/V)
    const int r = fdiv(idx, p.div_qg);
    x = idx - r * p.n_qg;
    bh = fdiv(r, p.div_split);
    split = r - bh * p.n_split;
  }
  bh += p.bh0;
  split += p.split0;
  const int qg = p.qg_desc ? p.n_qg - 1 - x : x;
  row0 = qg * (128 * QT);
}

// a[i] for a tile index i known only at run time, as a select between
// registers (indexing the array would put it in local memory).
template <int QT>
__device__ __forceinline__ int pick(const int (&a)[QT], int i) {
  if constexpr (QT == 1) return a[0];
  else return i == 0 ? a[0] : a[1];
}

// Item `idx` of the launch (idx < n_items): coordinates and the steps of each
// query tile.
template <int BC, int QT>
__device__ __forceinline__ void make_item(int idx, const FwdParams& p, Item<QT>& it) {
  item_coords<QT>(idx, p, it.bh, it.split, it.row0);
  const int kv_begin = it.split * p.tiles_per_split;
  const int kv_end = min(p.kv_tiles, kv_begin + p.tiles_per_split);
  // K/V tiles [b_i, e_i) of this split hold keys visible to rows of query
  // tile i (empty: e_i = b_i).  The item streams from cta_b = min b_i; tile i
  // takes steps [0, n_i), n_i = e_i - cta_b (its leading tiles before b_i are
  // fully masked for it and cost one MMA pair each).
  const int off = p.Nk - p.Nq;
  int cta_b = kv_end, kv_end_cta = kv_begin;
  bool any_tile = false;  // a split past the last K/V tile has kv_begin >= kv_end
#pragma unroll
  for (int i = 0; i < QT; ++i) {
    const int r_first = it.row0 + 128 * i;
    it.n[i] = -1;  // end tile, -1 = none
    if (r_first < p.Nq) {
      const int r_last = min(r_first + 128, p.Nq) - 1;
      // |r + off| < 2^30 and wl, wr <= 2^30: these sums stay within int
      const int klo = p.wl < 0 ? 0 : max(0, r_first + off - p.wl);
      const int khi = p.wr < 0 ? p.Nk - 1 : min(p.Nk - 1, r_last + off + p.wr);
      if (khi >= klo) {
        const int b = max(kv_begin, static_cast<int>(klo / BC));
        const int e = min(kv_end, static_cast<int>(khi / BC) + 1);
        if (e > b) {
          it.n[i] = e;
          any_tile = true;
          cta_b = min(cta_b, b);
          kv_end_cta = max(kv_end_cta, e);
        }
      }
    }
  }
  if (!any_tile) cta_b = kv_end_cta = kv_begin;  // nothing to stream
#pragma unroll
  for (int i = 0; i < QT; ++i) it.n[i] = it.n[i] < 0 ? 0 : it.n[i] - cta_b;
  it.cta_b = cta_b;
  it.n_cta = kv_end_cta - cta_b;
}

// Ring positions an item takes: its K and V tiles, plus (with O staged in
// ring slots) one slot per tile for the epilogue when it writes bf16 O of any
// tile; tile i's slot is position 2 n_cta + i.
template <bool kSlotStg, int QT>
__device__ __forceinline__ int item_positions(const Item<QT>& it, const FwdParams& p, bool& oslot) {
  oslot = false;
  if (kSlotStg && !p.partial)
#pragma unroll
    for (int i = 0; i < QT; ++i) oslot = oslot || it.n[i] > 0;
  return 2 * it.n_cta + (oslot ? QT : 0);
}

// Item of this CTA in round r (snake order), or -1 past the end.
__device__ __forceinline__ int item_of_round(int r, const FwdParams& p) {
  const int G = gridDim.x, c = blockIdx.x;
  const long long idx = static_cast<long long>(r) * G + ((r & 1) ? G - 1 - c : c);
  return idx < p.n_items ? static_cast<int>(idx) : -1;
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
  uint8_t* sStg = sQ + QT * C::kQTileBytes;  // own O staging (kOwnStg)
  uint8_t* sKV = sStg + (C::kOwnStg ? QT * C::kStgBytes : 0);
  Ctl* ctl = reinterpret_cast<Ctl*>(sKV + C::kStages * C::kKVTileBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rounds = p.rounds;

  const uint32_t bar_qf = smem_u32(&ctl->q_full[0]);
  const uint32_t bar_qe = smem_u32(&ctl->q_free[0]);
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
    for (int i = 0; i < QT; ++i) {
      mbar_init(bar_qf + 8 * i, 1);
      mbar_init(bar_qe + 8 * i, 1);
    }
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
    mbar_init(smem_u32(&ctl->stagger), 128);
    ctl->abort = 0;
    ctl->corr_stop[0] = ctl->corr_stop[1] = 0;
    fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
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
      // Per stage s, bits 2s + i: tile i reads the stage's current content
      // (rd), and the parity of the next kv_empty[s][i] phase to wait for (pe).
      uint32_t rd = 0, pe = 0;
      uint32_t filled = 0, fill_par = 0;  // per stage: ever filled; parity of its last fill
      int q_loads[QT];                    // Q_i loads so far
#pragma unroll
      for (int i = 0; i < QT; ++i) q_loads[i] = 0;
      int g_stage = 0;
      uint32_t g_par = 0;
      int g = 0;  // ring positions so far (the test hook counts these; stops at 2^31 - 1)
      bool ok = true;
      for (int r = 0; ok && r < rounds; ++r) {
        const int idx = item_of_round(r, p);
        if (idx < 0) continue;
        Item<QT> it;
        make_item<BC, QT>(idx, p, it);
        // Warm L2 with the next item's Q tiles, once this item's first loads
        // are under way (a prefetch occupies the TMA unit like a load).
        auto prefetch_next_q = [&]() {
          int nidx = -1;
          for (int r2 = r + 1; nidx < 0 && r2 < rounds; ++r2) nidx = item_of_round(r2, p);
          if (nidx >= 0) {
            int nbh, nsplit, nrow0;
            item_coords<QT>(nidx, p, nbh, nsplit, nrow0);
#pragma unroll
            for (int i = 0; i < QT; ++i)
              if (nrow0 + C::kBr * i < p.Nq)
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                  tma_prefetch_l2_3d(&tm_q, c * C::kChunkElems, nrow0 + C::kBr * i, nbh);
          }
        };
        // Q_i of this item, once the previous item's last S_i product is done.
        auto load_q = [&]() {
#pragma unroll
          for (int i = 0; i < QT; ++i) {
            if (it.n[i] <= 0) continue;
            if (q_loads[i] > 0 && !wait_bounded(bar_qe + 8 * i, (q_loads[i] - 1) & 1, wc)) return false;
            const uint32_t full = bar_qf + 8 * i;
            if (FA_DCHECK(it.bh < p.BH && it.row0 + C::kBr * i < p.Nq, p.status)) {
              mbar_arrive_expect_tx(full, C::kQTileBytes);
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(smem_u32(sQ + i * C::kQTileBytes + c * C::kQChunkBytes), &tm_q, full,
                            c * C::kChunkElems, it.row0 + C::kBr * i, it.bh);
            }
            ++q_loads[i];
          }
          return true;
        };
        bool oslot;
        const int n_pos = item_positions<C::kSlotStg, QT>(it, p, oslot);
        const int n_kv = 2 * it.n_cta;
        const int pf_at = min(n_kv, C::kStages + 1);
        if (!(ok = load_q())) break;
        for (int pos = 0; ok && pos < n_pos; ++pos) {
          if (pos == pf_at) prefetch_next_q();
          const RingPos rp = ring_at<C::kStages>(g_stage, g_par, pos);
          const int s2 = 2 * rp.stage;
          // the slot's previous content must be released by every tile that read it
#pragma unroll
          for (int i = 0; i < QT; ++i)
            if (ok && ((rd >> (s2 + i)) & 1u)) {
              ok = wait_bounded(bar_kv_empty + 16 * rp.stage + 8 * i, (pe >> (s2 + i)) & 1u, wc);
              pe ^= 1u << (s2 + i);
            }
          if (!ok) break;
          if (pos >= n_kv) {
            // O staging slot of tile pos - n_kv: no copy; that tile releases
            // it if it stages O
            const int ti = pos - n_kv;
            if (!FA_DCHECK(rp.stage < C::kStages && ti < QT, p.status)) continue;
            uint32_t stager = 0;
#pragma unroll
            for (int i = 0; i < QT; ++i) stager |= (i == ti && it.n[i] > 0 ? 1u : 0u) << i;
            rd = (rd & ~(3u << s2)) | (stager << s2);
            mbar_arrive(bar_kv_full + 8 * rp.stage);
            filled |= 1u << rp.stage;
            fill_par = (fill_par & ~(1u << rp.stage)) | (rp.par << rp.stage);
            continue;
          }
          bool is_v;
          int step;
          ring_decode(pos, it.n_cta, is_v, step);
          uint32_t readers = 0;
#pragma unroll
          for (int i = 0; i < QT; ++i) readers |= (step < it.n[i] ? 1u : 0u) << i;
          rd = (rd & ~(3u << s2)) | (readers << s2);
          const bool skip = g == p.test_skip_load;
          if (g < 0x7fffffff) ++g;
          if (skip) continue;  // test hook: this slot never fills
          const uint32_t full = bar_kv_full + 8 * rp.stage;
          if (!FA_DCHECK(rp.stage < C::kStages && step < it.n_cta && (it.cta_b + step) * BC < p.Nk &&
                             it.bh < p.BH,
                         p.status))
            continue;
          mbar_arrive_expect_tx(full, C::kKVTileBytes);
          const CUtensorMap* map = is_v ? &tm_v : &tm_k;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem_u32(sKV + rp.stage * C::kKVTileBytes + c * C::kKVChunkBytes), map, full,
                        c * C::kChunkElems, (it.cta_b + step) * BC, it.bh);
          filled |= 1u << rp.stage;
          fill_par = (fill_par & ~(1u << rp.stage)) | (rp.par << rp.stage);
        }
        ring_advance<C::kStages>(g_stage, g_par, n_pos);
      }
      // Every copy started here must land before the CTA may exit.
      for (int s = 0; s < C::kStages; ++s)
        if ((filled >> s) & 1u) wait_own(bar_kv_full + 8 * s, (fill_par >> s) & 1u, p.timeout_ns);
#pragma unroll
      for (int i = 0; i < QT; ++i)
        if (q_loads[i] > 0) wait_own(bar_qf + 8 * i, (q_loads[i] - 1) & 1, p.timeout_ns);
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
      // Phases carried across items: S products of this tile and of the other
      // one so far (= the s_free / pv_ready / o_done phases), Q_i loads
      // consumed, the ring base, and the last product in a shared S buffer.
      int cs_me = 0, cs_ot = 0;
      int q_loads = 0;
      int g_stage = 0;
      uint32_t g_par = 0;
      int last_t = -1, last_c = 0;
      int stag = 0;  // stagger phases waited for (tile 1)
      // debug build: this tile's TMEM columns lie inside the allocation
      bool ok = FA_DCHECK(i < QT && (tmem & 0xFFFFu) + C::kTmemNeed <= 512u, p.status), issued = false;
      for (int r = 0; ok && r < rounds; ++r) {
        const int idx = item_of_round(r, p);
        if (idx < 0) continue;
        Item<QT> it;
        make_item<BC, QT>(idx, p, it);
        const int n = pick<QT>(it.n, i);
        const int n_ot = QT == 2 ? pick<QT>(it.n, 1 - i) : 0;
        const int n_cta = it.n_cta;
        auto kv_ready = [&](int pos) {
          const RingPos rp = ring_at<C::kStages>(g_stage, g_par, pos);
          return warp_wait(bar_kv_full + 8 * rp.stage, rp.par, wc);
        };
        // A shared S buffer is taken in the order S_0(0), S_1(0), S_0(1), ...
        // (a tile past its last step drops out), continuing from the previous
        // item's last product; a tile's own buffer holds S_i(0), S_i(1), ...
        // Each use waits until the previous one has been read into registers.
        auto prev_use = [&](int q, uint32_t& bar, uint32_t& par) {
          if constexpr (QT == 2 && C::kSharedS) {
            const int o = 1 - i, qo = i == 1 ? q : q - 1;
            if (qo >= 0 && qo < n_ot) {
              bar = bar_sfree + 8 * o, par = (cs_ot + qo) & 1;
              return true;
            }
            if (q == 0) {
              if (last_t < 0) return false;
              bar = bar_sfree + 8 * last_t, par = last_c & 1;
              return true;
            }
          } else {
            if (q == 0) {
              if (cs_me == 0) return false;
              bar = bar_sfree + 8 * i, par = (cs_me - 1) & 1;
              return true;
            }
          }
          bar = bar_sfree + 8 * i, par = (cs_me + q - 1) & 1;
          return true;
        };
        auto s_ready = [&](int q) {  // S_i(q) may be written: the buffer's previous product was read
          uint32_t bar, par;
          return !prev_use(q, bar, par) || warp_wait(bar, par, wc);
        };
        auto issue_qk = [&](int q) {  // S_i(q) = Q_i K_q^T, then release K_q's slot for tile i
          const int stage = ring_at<C::kStages>(g_stage, g_par, ring_pos_k(q)).stage;
          if (!FA_DCHECK(stage < C::kStages && q < n, p.status)) return;
          const uint32_t k_lo = lo_k + ((stage * C::kKVTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / C::kKStep; ++kk) {  // 32 bytes of K per step
            const uint32_t off_q = ((kk / 4) * C::kQChunkBytes + (kk % 4) * 32) >> 4;
            const uint32_t off_k = ((kk / 4) * C::kKVChunkBytes + (kk % 4) * 32) >> 4;
            mma(tS, hi_q | (lo_q + off_q), hi_k | (k_lo + off_k), kIdescQK, kk > 0);
          }
          mma_commit_elect(bar_s + 8 * i);
          mma_commit_elect(bar_kv_empty + 16 * stage + 8 * i);
          // After this item's last S_i, Q_i may be overwritten.
          if (q == n - 1) mma_commit_elect(bar_qe + 8 * i);
        };
        auto issue_pv = [&](int v) {  // O_i += P_i(v) V_v, then release V_v's slot for tile i
          const int stage = ring_at<C::kStages>(g_stage, g_par, ring_pos_v(v, n_cta)).stage;
          if (!FA_DCHECK(stage < C::kStages && v < n, p.status)) return;
          const uint32_t v_lo = lo_v + ((stage * C::kKVTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < BC / C::kKStep; ++kk) {
            // P: one K-step (32 bytes = 8 TMEM columns of packed P).  V: kKStep
            // keys = 8-row groups of 1024 B (SBO); D columns in 128-byte chunks
            // BC*128 B apart (LBO).  The item's first product overwrites O_i.
            mma_ts(tO, tP + 8 * kk, hi_v | (v_lo + ((kk * C::kKStep * 128) >> 4)), kIdescPV,
                   (v > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_elect(bar_o + 8 * i);
          mma_commit_elect(bar_kv_empty + 16 * stage + 8 * i);
        };
        if (n > 0) {
          // S_i(j+1) first: it waits only for the other tile to read its S,
          // which comes before P_i(j) is ready.
          ok = warp_wait(bar_qf + 8 * i, q_loads & 1, wc) && s_ready(0) && kv_ready(ring_pos_k(0));
          ++q_loads;
          if constexpr (C::kStagger) {
            if (i == 1 && n_ot > 0) {
              ok = ok && warp_wait(smem_u32(&ctl->stagger), stag & 1, wc);
              ++stag;
            }
          }
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
            ok = warp_wait(bar_pv + 8 * i, (cs_me + j) & 1, wc) && kv_ready(ring_pos_v(j, n_cta));
            if (!ok) break;
            tc_fence_after();
            issue_pv(j);
          }
        }
        if constexpr (QT == 2 && C::kSharedS) {
          // tile 1's last product comes last unless tile 0 has more steps
          const int n0 = i == 0 ? n : n_ot, n1 = i == 0 ? n_ot : n;
          const int c0 = i == 0 ? cs_me : cs_ot, c1 = i == 0 ? cs_ot : cs_me;
          if (n0 > 0 || n1 > 0) {
            if (n1 >= n0) {
              last_t = 1, last_c = c1 + n1 - 1;
            } else {
              last_t = 0, last_c = c0 + n0 - 1;
            }
          }
        }
        cs_me += n;
        cs_ot += n_ot;
        bool oslot;
        ring_advance<C::kStages>(g_stage, g_par, item_positions<C::kSlotStg, QT>(it, p, oslot));
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
    // let the MMA warp issue O_i += P_i(j) V_j.  Steps are counted from the
    // start of the CTA across its items; an item's first step publishes
    // alpha = 1 (its first product overwrites O_i), so item boundaries need
    // no handling here.  After its last item, tile i publishes one more
    // alpha phase with corr_stop[i] set: that tile is finished.
    if constexpr (C::kSplitRegs && C::kRegCorr < C::kRegLaunch) setmaxnreg_dec<C::kRegCorr>();
    const int t = threadIdx.x & 127;
    int jn[QT];     // next step of tile i
    bool have[QT];  // alpha_i(jn) read, waiting for the previous P.V
    bool fin[QT];   // tile i finished
    float alpha_r[QT];
#pragma unroll
    for (int i = 0; i < QT; ++i) {
      jn[i] = 0;
      have[i] = false;
      fin[i] = false;
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
        if (fin[i]) continue;
        done = false;
        if (!have[i]) {
          if (!probe(bar_alpha + 8 * i, j & 1)) {
            continue;
          }
          if (*reinterpret_cast<volatile int*>(&ctl->corr_stop[i])) {
            fin[i] = true;
            progressed = true;
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
            record_status(p.status, kDevTimeout);
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
    const float c = p.scale_log2;
    const int off = p.Nk - p.Nq;
    int cs = 0;            // steps of this tile in earlier items (s_full, pv_ready, o_done phases)
    bool stg_pending = false;  // thread 0: a TMA store from the staging buffer may still read it
    uint32_t g_sp = 0;     // ring position of the item's first K tile: stage | parity << 8
    // debug build: this tile's TMEM columns lie inside the allocation
    const int my_rounds =
        FA_DCHECK(i < QT && (tmem & 0xFFFFu) + C::kTmemNeed <= 512u, p.status) ? rounds : 0;
    for (int r = 0; r < my_rounds; ++r) {
      const int idx = item_of_round(r, p);
      if (idx < 0) continue;
      // Only what the step loop needs stays live through it; the epilogue
      // decodes the item again.
      int n, cta_b, row0;
      bool stagger = false;  // tile 0 releases tile 1's first S product of the item
      {
        Item<QT> it;
        make_item<BC, QT>(idx, p, it);
        n = pick<QT>(it.n, i);
        cta_b = it.cta_b;
        row0 = it.row0 + C::kBr * i;  // first row of this tile
        if constexpr (C::kStagger) stagger = i == 0 && it.n[1] > 0;
      }
      const int row = row0 + t;
      // The row sits at key position rq = row + Nk - Nq; keys visible to it are
      // [rq - wl, rq + wr] within [0, Nk), a -1 bound leaving that side open.
      // (|rq| < 2^30 and wl, wr <= 2^30, so the sums below stay within int.)
      // K/V tiles [jf_b, jf_e) hold only keys that every row of this query tile
      // sees; they skip the mask (a test uniform across the warpgroup).
      const int rq = row + off;
      int jf_b = 0, jf_e;
      {
        const int tr_first = row0 + off;
        const int tr_last = min(row0 + C::kBr, p.Nq) - 1 + off;
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
        if (!warp_wait(bar_s + 8 * i, (cs + jj) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();

        uint32_t rg[BC];
        if constexpr (BC == 128)
          tmem_ld64x2_sync(tS, tS + 64, rg);
        else
          tmem_ld64_sync(tS, rg);
        tc_fence_before();
        mbar_arrive(bar_sfree + 8 * i);  // the S buffer may take the next product
        float s[BC];
#pragma unroll
        for (int cc = 0; cc < BC; ++cc) s[cc] = __uint_as_float(rg[cc]);
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
        if constexpr (C::kStagger) {
          if (stagger && jj == 0) mbar_arrive(smem_u32(&ctl->stagger));
        }
        const bool bump = mt > m && (m == -INFINITY || (mt - m) * c > C::kLazy);
        const float m_new = bump ? mt : m;
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = bump ? ex2_approx((m - m_ref) * c) : 1.f;
        if constexpr (C::kCorr) {
          // The correction must have read the previous alpha_i before the slot
          // is reused (S_i(j) was issued before it ran, so this step can be
          // ahead of it).
          if (cs + jj > 0 && !warp_wait(bar_afree + 8 * i, (cs + jj - 1) & 1, wc)) {
            ok = false;
            break;
          }
          // the correction warpgroup rescales O_i by it (not at an item's
          // first step: that product overwrites O_i)
          ctl->alpha[i][t] = jj == 0 ? 1.f : alpha;
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
        if (jj > 0 && !warp_wait(bar_o + 8 * i, (cs + jj - 1) & 1, wc)) {
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
      if (ok && n > 0) ok = warp_wait(bar_o + 8 * i, (cs + n - 1) & 1, wc);
      cs += n;
      Item<QT> it;
      make_item<BC, QT>(idx, p, it);
      const int bh = it.bh;
      // this tile's O staging slot (after the item's K/V tiles), then the next
      // item's ring base
      RingPos slot;
      {
        int g_stage = static_cast<int>(g_sp & 0xffu);
        uint32_t g_par = g_sp >> 8;
        slot = ring_at<C::kStages>(g_stage, g_par, 2 * it.n_cta + i);
        bool oslot;
        ring_advance<C::kStages>(g_stage, g_par, item_positions<C::kSlotStg, QT>(it, p, oslot));
        g_sp = static_cast<uint32_t>(g_stage) | (g_par << 8);
      }
      // The previous item's O store must have read the staging buffer before
      // it is written again (the barrier below orders that for the others).
      if (C::kOwnStg && stg_pending && t == 0) {
        tma_store_wait_read();
        stg_pending = false;
      }
      const bool bad = named_bar_or(1 + i, 128, !ok || *wc.abort);
      if (bad) break;
      // A tile that starts past the last query row has nothing to write.
      if (row0 >= p.Nq) continue;
      if (n > 0) tc_fence_after();
      const bool empty = !(l > 0.f);
      // FP8: sum_scale l <- l 2^-8 undoes Max_offset in the row sum, and
      // final_scale (p.o_scale = v_descale 2^-8) in O ("Online Softmax 算法详解"
      // section 6.3); both are powers of two or exact scalings.
      const float lc = F8 ? l * (1.f / 256.f) : l;
      const float inv = empty ? 0.f : (F8 ? p.o_scale / lc : 1.f / (l + l_fix));
      if (!p.partial) {
        if (n == 0) {
          // no visible key: O = 0 straight to global memory (the staging
          // buffers may be in use by the next item's loads)
          if (row < p.Nq && FA_DCHECK(bh < p.BH, p.status)) {
            uint8_t* orow = static_cast<uint8_t*>(p.o) + (static_cast<size_t>(bh) * p.Nq + row) * (D * 2);
#pragma unroll
            for (int q = 0; q < D * 2 / 16; ++q) st_global_v4(orow + 16 * q, 0u, 0u, 0u, 0u);
          }
        } else {
          // bf16 O, staged with the 128-byte swizzle, then TMA stores (rows past
          // Nq are clipped by the map): all of O at once in the tile's ring
          // slot, or 64 columns per round through its own 16 KB buffer.
          uint32_t stg;
          constexpr int kRounds = C::kSlotStg ? 1 : D / 64;
          if constexpr (C::kSlotStg) {
            // every warp of the tile agrees before any of them leaves
            const bool got = FA_DCHECK(slot.stage < C::kStages && bh < p.BH, p.status) &&
                             warp_wait(bar_kv_full + 8 * slot.stage, slot.par, wc);
            if (named_bar_or(1 + i, 128, !got)) break;
            stg = smem_u32(sKV + slot.stage * C::kKVTileBytes);
          } else {
            stg = smem_u32(sStg + i * C::kStgBytes);
          }
#pragma unroll
          for (int round = 0; round < kRounds; ++round) {
            if (round > 0) {  // staging buffer free again
              if (t == 0) tma_store_wait_read();
              named_bar_sync(1 + i, 128);
            }
#pragma unroll
            for (int ch = 0; ch < D / 64 / kRounds; ++ch) {  // 64-column chunks of this round
              const int col = (round * (D / 64 / kRounds) + ch) * 64;
              uint32_t o[64];
              tmem_ld64_sync(tO + col, o);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                uint32_t wv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  wv[k] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * k]) * inv,
                                      __uint_as_float(o[8 * q + 2 * k + 1]) * inv);
                st_shared_v4(stg + ch * C::kStgBytes + t * 128 + ((q ^ (t & 7)) << 4), wv[0], wv[1],
                             wv[2], wv[3]);
              }
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + i, 128);
            if (t == 0) {
#pragma unroll
              for (int ch = 0; ch < D / 64 / kRounds; ++ch)
                tma_store_3d(&tm_o, stg + ch * C::kStgBytes, (round * (D / 64 / kRounds) + ch) * 64, row0, bh);
              tma_store_commit();
            }
          }
          if (t == 0) {
            if constexpr (C::kOwnStg) {
              stg_pending = true;  // waited for before the next use
            } else {
              tma_store_wait_read();
              mbar_arrive(bar_kv_empty + 16 * slot.stage + 8 * i);  // the slot goes back to the ring
            }
          }
        }
        if (row < p.Nq && FA_DCHECK(bh < p.BH, p.status))
          p.lse[static_cast<size_t>(bh) * p.Nq + row] = empty ? -INFINITY : m * p.scale + logf(lc);
      } else {
        // fp32 partial triple (m in natural-log units, l, O/l) for the merge.
        const size_t prow = (static_cast<size_t>(it.split) * p.BH + bh) * p.Nq + row;
        if (!FA_DCHECK(it.split < p.n_splits && bh < p.BH, p.status)) continue;
        if (row < p.Nq) {
          p.m_part[prow] = empty ? -INFINITY : m * p.scale;
          p.l_part[prow] = empty ? 0.f : l;
        }
        // O/l in fp32 (fa_fwd_partial), or rounded to bf16 (fa_fwd's own
        // split workspace: half the bytes through HBM on both sides of the merge)
        const bool bf = p.part_bf16 != 0;
        uint8_t* op = static_cast<uint8_t*>(p.o_part) + prow * (D * (bf ? 2 : 4));
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
            if (bf) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  w[k] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * k]), __uint_as_float(o[8 * q + 2 * k + 1]));
                st_global_v4(op + 2 * cc + 16 * q, w[0], w[1], w[2], w[3]);
              }
            } else {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_global_v4(op + 4 * cc + 16 * q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
          }
        }
      }
    }
    if (C::kOwnStg && stg_pending && t == 0) tma_store_wait_read();
    if constexpr (C::kCorr) {
      // Tell the correction this tile is finished: one more alpha phase, with
      // the stop flag set, once it has read the last alpha.
      const bool ok2 = !*wc.abort && (cs == 0 || warp_wait(bar_afree + 8 * i, (cs - 1) & 1, wc));
      if (!named_bar_or(1 + i, 128, !ok2)) {
        if (t == 0) *reinterpret_cast<volatile int*>(&ctl->corr_stop[i]) = 1;
        mbar_arrive(bar_alpha + 8 * i);  // after the flag store (release)
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
