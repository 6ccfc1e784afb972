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
// (the whole key axis, or one split of it).  Warp roles:
//   warps 0 .. 4*QT-1   softmax warpgroup i = warp/4 owns Q tile i; thread t
//                       owns row t of that tile (TMEM lane t), so row max and
//                       row sum are register-local (no shuffles).  Also does
//                       the O rescale and the epilogue of its tile.
//   warp 4*QT           MMA issuer (one elected thread).
//   warp 4*QT+1         TMA producer (one elected thread): Q once, then K_j,
//                       V_j, K_{j+1}, ... through a ring of shared-memory stages.
// TMEM (fp32 columns): S_i at [i*BC, (i+1)*BC), O_i at [QT*BC + i*D, ..+D).
// P_i (bf16 pairs) overwrites the first BC/2 columns of S_i and is the A
// operand of the P.V MMA straight from TMEM.  Because P_i aliases S_i, the
// MMA thread issues S_i(j+1) only after P_i(j).V_j has completed.
//
// Every mbarrier wait is bounded by a global-timer limit.  A wait that runs
// out sets the CTA's abort flag and the device status word; every role then
// leaves its loop, lets its own copies / MMAs in flight finish, and the CTA
// frees TMEM and exits without writing outputs.
#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D, int BC, int QT>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BC == 64 || BC == 128, "K/V tile");
  static_assert(QT == 1 || QT == 2, "Q tiles per CTA");
  static constexpr int kBr = 128;  // query rows per tile (= TMEM lanes)
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kLoadWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  static constexpr int kChunks = D / 64;         // 64-column (128-byte) swizzle chunks
  static constexpr int kQChunkBytes = kBr * 128;  // 128 rows x 128 B
  static constexpr int kQTileBytes = kChunks * kQChunkBytes;
  static constexpr int kKVChunkBytes = BC * 128;
  static constexpr int kKVTileBytes = kChunks * kKVChunkBytes;
  static constexpr int kSCol = 0;
  static constexpr int kOCol = QT * BC;
  static constexpr int kTmemNeed = QT * (BC + D);
  static constexpr int kTmemCols = kTmemNeed <= 64    ? 64
                                   : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256
                                                      : 512;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int kStagesFit =
      (kSmemLimit - 1024 - kCtlBytes - QT * kQTileBytes) / kKVTileBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static_assert(kStages >= 2, "shared memory");
  static constexpr int kSmemBytes = 1024 + QT * kQTileBytes + kStages * kKVTileBytes + kCtlBytes;
};

struct __align__(8) Ctl {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct WaitCtx {
  volatile int* abort;
  int* status;
  unsigned long long timeout_ns;
};

// Bounded wait on a phase; false if the CTA aborted or the limit ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.timeout_ns) {
      *w.abort = 1;
      atomicExch(w.status, kDevTimeout);
      return false;
    }
  }
}

// Bounded wait for this thread's own copies / MMAs in flight (ignores abort).
__device__ __forceinline__ void wait_own(uint32_t bar, uint32_t parity,
                                         unsigned long long timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

template <int D, int BC, int QT>
__global__ void __launch_bounds__(FwdCfg<D, BC, QT>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using C = FwdCfg<D, BC, QT>;
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
  int end_i[QT];
  int kv_end_cta = kv_begin;
#pragma unroll
  for (int i = 0; i < QT; ++i) {
    const int r_first = row0 + C::kBr * i;
    int e = kv_begin;
    if (r_first < p.Nq) {
      e = kv_end;
      if (p.causal) {
        // last key visible to the tile's last row: r_last + (Nk - Nq)
        const int r_last = min(r_first + C::kBr, p.Nq) - 1;
        const long long last_key = static_cast<long long>(r_last) + (p.Nk - p.Nq);
        const int lim = last_key < 0 ? 0 : static_cast<int>(last_key / BC) + 1;
        e = min(e, lim);
      }
      e = max(e, kv_begin);
    }
    end_i[i] = e;
    kv_end_cta = max(kv_end_cta, e);
  }

  const uint32_t bar_q = smem_u32(&ctl->q_full);
  const uint32_t bar_kv_full = smem_u32(&ctl->kv_full[0]);
  const uint32_t bar_kv_empty = smem_u32(&ctl->kv_empty[0]);
  const uint32_t bar_s = smem_u32(&ctl->s_full[0]);
  const uint32_t bar_p = smem_u32(&ctl->p_full[0]);
  const uint32_t bar_o = smem_u32(&ctl->o_done[0]);
  const uint32_t bar_drain = smem_u32(&ctl->drain);

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full + 8 * s, 1);
      mbar_init(bar_kv_empty + 8 * s, 1);
    }
    for (int i = 0; i < QT; ++i) {
      mbar_init(bar_s + 8 * i, 1);
      mbar_init(bar_p + 8 * i, 128);
      mbar_init(bar_o + 8 * i, 1);
    }
    mbar_init(bar_drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const WaitCtx wc{&ctl->abort, p.status, p.timeout_ns};

  if (warp == C::kLoadWarp) {
    // ================================================================ producer
    if (lane == 0) {
      uint32_t qbytes = 0;
#pragma unroll
      for (int i = 0; i < QT; ++i)
        if (end_i[i] > kv_begin) qbytes += C::kQTileBytes;
      if (qbytes) {
        mbar_arrive_expect_tx(bar_q, qbytes);
#pragma unroll
        for (int i = 0; i < QT; ++i) {
          if (end_i[i] <= kv_begin) continue;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem_u32(sQ + i * C::kQTileBytes + c * C::kQChunkBytes), &tm_q, bar_q,
                        c * 64, row0 + C::kBr * i, bh);
        }
      }
      uint32_t issued_mask = 0, issued_par = 0;
      int it = 0;
      bool ok = true;
      for (int j = kv_begin; ok && j < kv_end_cta; ++j) {
        for (int kv = 0; kv < 2; ++kv, ++it) {
          const int stage = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!wait_bounded(bar_kv_empty + 8 * stage, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          if (it == p.test_skip_load) continue;  // test hook: this stage never fills
          const uint32_t full = bar_kv_full + 8 * stage;
          mbar_arrive_expect_tx(full, C::kKVTileBytes);
          const CUtensorMap* map = kv ? &tm_v : &tm_k;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem_u32(sKV + stage * C::kKVTileBytes + c * C::kKVChunkBytes), map, full,
                        c * 64, j * BC, bh);
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (ph << stage);
        }
      }
      // Every copy started here must land before the CTA may exit.
      for (int s = 0; s < C::kStages; ++s)
        if ((issued_mask >> s) & 1u) wait_own(bar_kv_full + 8 * s, (issued_par >> s) & 1u, p.timeout_ns);
      if (qbytes) wait_own(bar_q, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, BC, false);  // K-major A (Q), B (K)
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);    // B = V is MN-major
      bool ok = kv_end_cta > kv_begin;
      if (ok) ok = wait_bounded(bar_q, 0, wc);
      if (ok) tc_fence_after();
      int it = 0;
      for (int jj = 0; ok && kv_begin + jj < kv_end_cta; ++jj) {
        const int j = kv_begin + jj;
        {  // S_i = Q_i K_j^T
          const int stage = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          ++it;
          if (!wait_bounded(bar_kv_full + 8 * stage, ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sK = smem_u32(sKV + stage * C::kKVTileBytes);
#pragma unroll
          for (int i = 0; i < QT; ++i) {
            if (j >= end_i[i]) continue;
            if (jj > 0) {  // P_i(j-1) (aliasing S_i) must have been consumed
              if (!wait_bounded(bar_o + 8 * i, (jj - 1) & 1, wc)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t sQi = smem_u32(sQ + i * C::kQTileBytes);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off_q = (kk / 4) * C::kQChunkBytes + (kk % 4) * 32;
              const uint32_t off_k = (kk / 4) * C::kKVChunkBytes + (kk % 4) * 32;
              mma_bf16_ss(tmem + C::kSCol + i * BC, smem_desc_sw128(sQi + off_q, 16, 1024),
                          smem_desc_sw128(sK + off_k, 16, 1024), kIdescQK, kk > 0);
            }
            mma_commit(bar_s + 8 * i);
          }
          if (!ok) break;
          mma_commit(bar_kv_empty + 8 * stage);
        }
        {  // O_i += P_i V_j
          const int stage = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          ++it;
          if (!wait_bounded(bar_kv_full + 8 * stage, ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sV = smem_u32(sKV + stage * C::kKVTileBytes);
#pragma unroll
          for (int i = 0; i < QT; ++i) {
            if (j >= end_i[i]) continue;
            if (!wait_bounded(bar_p + 8 * i, jj & 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BC / 16; ++kk) {
              // 16 keys = two 8-row groups (SBO 1024 B); D columns in 64-wide
              // chunks BC*128 B apart (LBO).
              mma_bf16_ts(tmem + C::kOCol + i * D, tmem + C::kSCol + i * BC + kk * 8,
                          smem_desc_sw128(sV + kk * 2048, C::kKVChunkBytes, 1024), kIdescPV,
                          (jj > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar_o + 8 * i);
          }
          if (!ok) break;
          mma_commit(bar_kv_empty + 8 * stage);
        }
      }
      // Everything issued above completes before TMEM may be freed.
      mma_commit(bar_drain);
      wait_own(bar_drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ===================================================== softmax warpgroup
    const int i = warp >> 2;
    const int t = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kSCol + i * BC;
    const uint32_t tO = tmem + lane_off + C::kOCol + i * D;
    const int row = row0 + C::kBr * i + t;
    const int n = end_i[i] - kv_begin;
    const float c = p.scale_log2;
    // last key visible to this row
    const int lim = p.causal ? min(p.Nk - 1, row + (p.Nk - p.Nq)) : p.Nk - 1;
    float m = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int jj = 0; jj < n; ++jj) {
      const int j = kv_begin + jj;
      bool got = wait_bounded(bar_s + 8 * i, jj & 1, wc);
      if (got && jj > 0) got = wait_bounded(bar_o + 8 * i, (jj - 1) & 1, wc);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();

      uint32_t r[BC];
#pragma unroll
      for (int h = 0; h < BC / 64; ++h) tmem_ld64_sync(tS + h * 64, r + h * 64);
      float s[BC];
#pragma unroll
      for (int cc = 0; cc < BC; ++cc) s[cc] = __uint_as_float(r[cc]);
      const int key0 = j * BC;
      if (key0 + BC - 1 > lim) {  // tail of the key axis or causal diagonal
#pragma unroll
        for (int cc = 0; cc < BC; ++cc)
          if (key0 + cc > lim) s[cc] = -INFINITY;
      }

      // m' = max(m, rowmax S): eight independent partial maxima
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = s[u];
#pragma unroll
      for (int cc = 8; cc < BC; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], s[cc]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m, mt);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_new == m) ? 1.f : ex2_approx((m - m_ref) * c);

      // P = 2^(s*c - m_ref*c); rowsum of the fp32 P (before the bf16 cast)
      const float neg = m_ref * c;
      float ls[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) ls[u] = 0.f;
      uint32_t pk[BC / 2];
#pragma unroll
      for (int cc = 0; cc < BC; cc += 2) {
        const float p0 = ex2_approx(fmaf(s[cc], c, -neg));
        const float p1 = ex2_approx(fmaf(s[cc + 1], c, -neg));
        ls[(cc >> 1) & 7] += p0 + p1;
        pk[cc >> 1] = pack_bf16x2(p0, p1);
      }
      const float rowsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
#pragma unroll
      for (int h = 0; h < BC / 64; ++h) tmem_st32(tS + h * 32, pk + h * 32);

      // O <- alpha O (PV_i(j-1) is complete), skipped when no row of this
      // warp changed its max.
      if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32_sync(tO + cc, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tO + cc, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p + 8 * i);
      l = alpha * l + rowsum;
      m = m_new;
    }
    if (ok && n > 0) {
      const bool got = wait_bounded(bar_o + 8 * i, (n - 1) & 1, wc);
      ok = __all_sync(0xffffffffu, got);
    }
    const bool bad = named_bar_or(1 + i, 128, !ok || *wc.abort);
    // A tile that starts past the last query row has nothing to write.
    if (!bad && row0 + C::kBr * i < p.Nq) {
      if (n > 0) tc_fence_after();
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.f / l;
      if (!p.partial) {
        // bf16 O, staged in this tile's (now unused) Q buffer with the 128-byte
        // swizzle, then one TMA store (rows past Nq are clipped by the map).
        const uint32_t stg = smem_u32(sQ + i * C::kQTileBytes);
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
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
          const int chunk = cc / 64;
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
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_store_3d(&tm_o, stg + ch * C::kQChunkBytes, ch * 64, row0 + C::kBr * i, bh);
          tma_store_commit();
          tma_store_wait_read();
        }
        if (row < p.Nq)
          p.lse[static_cast<size_t>(bh) * p.Nq + row] = empty ? -INFINITY : m * p.scale + logf(l);
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
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int BC, int QT>
cudaError_t launch_fwd_t(const CUtensorMap* maps, const FwdParams& p, dim3 grid, cudaStream_t s) {
  using C = FwdCfg<D, BC, QT>;
  auto kern = fa_fwd_kernel<D, BC, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

}  // namespace fa
