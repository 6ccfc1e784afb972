// fa_softmax.cu -- softmax over the rows of a matrix with the online
// normaliser: pass 1 fuses the running max and the rescaled sum, pass 2
// normalises ("Online Softmax 算法详解" section 2.2, the two-pass scheme).
//
// Each thread owns a slice of the row (16-byte vectors, consecutive threads on
// consecutive vectors).  Over its slice it keeps the pair (m, l): per vector
// group, a new max rescales l by exp(m_old - m_new) and the group's
// exponentials are added against the new max; that is the recurrence applied
// to blocks of the row, exact for any partition ("在线Softmax算法解析" section
// 3.2).  The threads' pairs are then combined with the two-block merge rule
// (airsota.com online-softmax card, section 三) -- within a warp by shuffles,
// across warps through shared memory, and, when a thread-block cluster shares
// the row, across its CTAs through distributed shared memory -- always in the
// same order, so every CTA of a row gets the same (M, L).  Pass 2 writes
// y = exp(x - M) / L.
//
// A row that fits one CTA (up to 1024 threads x 16 fp32 or 32 bf16 values)
// runs fa_softmax_rows_kernel: 16-byte (or element) loads straight into
// registers, several CTAs per SM overlapping one another.  Longer rows with
// 16-byte aligned starts run fa_softmax_ring_kernel on a cluster of up to 8
// CTAs of 1024 threads: each CTA's columns of each row arrive through a ring
// of shared-memory stages filled by 1-D bulk copies (TMA) issued rows ahead,
// so loads overlap the arithmetic and the stores of earlier rows; the threads
// copy their slice into registers and free the stage at once.  Either way a
// row that fits the registers of its CTA or cluster is read from HBM once and
// pass 2 rescales the exponentials kept from pass 1 by exp(m_thread - M) / L.
// Longer rows are cut into sub-chunks and pass 2 streams them through the
// ring again; pass 1 marks them to stay in L2 for that second read.
//
// Exponentials: exp(x - m) = 2^((x - m) log2 e), the difference taken first
// (so the exponent's rounding error scales with |x - m|, not with |m|) and
// the power with ex2.approx.ftz; a running max of -inf uses 0 as its
// reference point, so no (-inf) - (-inf) appears ("Online Softmax 算法详解"
// section 7.1).  A row with no finite entry gets y = 0 and LSE = -inf.
#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_wait.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCluster = 8;

template <typename T>
struct Io;

template <>
struct Io<float> {
  static constexpr int E = 4;  // elements per 16-byte vector
  template <bool kKeepL2>
  __device__ static void load_vec(const float* p, float* v) {
    const float4 t = kKeepL2 ? __ldg(reinterpret_cast<const float4*>(p))
                             : __ldcs(reinterpret_cast<const float4*>(p));
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  }
  __device__ static float load_one(const float* p) { return __ldg(p); }
  __device__ static void store_vec(float* p, const float* v) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  }
  __device__ static void store_one(float* p, float v) { __stcs(p, v); }
};

template <>
struct Io<__nv_bfloat16> {
  static constexpr int E = 8;
  template <bool kKeepL2>
  __device__ static void load_vec(const __nv_bfloat16* p, float* v) {
    const uint4 t = kKeepL2 ? __ldg(reinterpret_cast<const uint4*>(p))
                            : __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bf16 -> fp32 is exact: the bits move up 16
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __device__ static float load_one(const __nv_bfloat16* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)))
                           << 16);
  }
  __device__ static void store_vec(__nv_bfloat16* p, const float* v) {
    uint4 t;
    t.x = pack_bf16x2(v[0], v[1]);
    t.y = pack_bf16x2(v[2], v[3]);
    t.z = pack_bf16x2(v[4], v[5]);
    t.w = pack_bf16x2(v[6], v[7]);
    __stcs(reinterpret_cast<uint4*>(p), t);
  }
  __device__ static void store_one(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// (m, l) <- (m, l) merged with (m2, l2): the two-block rule.  The pair with
// the larger max keeps its sum as is (its factor exp(0) is exactly 1), so one
// exponential suffices; a -inf max carries l = 0 and contributes nothing.
__device__ __forceinline__ void merge_pair(float& m, float& l, float m2, float l2) {
  if (m >= m2) {
    if (m2 != -INFINITY) l += l2 * ex2_approx((m2 - m) * kLog2e);
  } else {
    l = (m != -INFINITY ? l * ex2_approx((m - m2) * kLog2e) : 0.f) + l2;
    m = m2;
  }
}

// Tree of merges over the 32 lanes (fixed order); lane 0's pair is broadcast.
__device__ __forceinline__ float2 warp_pair(float m, float l) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_down_sync(0xffffffffu, m, o);
    const float l2 = __shfl_down_sync(0xffffffffu, l, o);
    merge_pair(m, l, m2, l2);
  }
  return make_float2(__shfl_sync(0xffffffffu, m, 0), __shfl_sync(0xffffffffu, l, 0));
}

// Every warp reduces its lanes, publishes its pair, and then reduces the
// warps' pairs itself -- the same tree in every warp, so every thread returns
// the same block pair after a single barrier.  `par` alternates by row: a
// warp writes row it's slot only after the barrier of row it-1, which every
// warp passes only once done reading row it-2's slots.
template <int kThreads>
__device__ __forceinline__ float2 block_pair(float m, float l, float2 (*warp_part)[kThreads / 32],
                                             int par) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 w = warp_pair(m, l);
  if (kWarps == 1) return w;
  if (lane == 0) warp_part[par][warp] = w;
  __syncthreads();
  const float2 b = lane < kWarps ? warp_part[par][lane] : make_float2(-INFINITY, 0.f);
  return warp_pair(b.x, b.y);
}

template <typename T, int kThreads, int kVec, bool kVecIO>
__global__ void __launch_bounds__(kThreads) fa_softmax_rows_kernel(const SoftmaxParams p) {
  using IO = Io<T>;
  constexpr int E = IO::E;
  constexpr int kPer = kVec * E;           // values a thread holds per sub-chunk
  constexpr int kSub = kThreads * kPer;    // columns per sub-chunk
  constexpr int kWarps = kThreads / 32;
  __shared__ float2 warp_part[2][kWarps];  // per-warp (m, l), double-buffered by row
  __shared__ float2 peer_part[2][kMaxCluster];  // written by every CTA of the cluster

  const int tid = threadIdx.x;
  const int ncta = p.cluster;
  const int rank = ncta > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const long long groups = gridDim.x / ncta;
  const long long group = blockIdx.x / ncta;
  const int c0 = rank * p.chunk;
  const int c1 = min(p.cols, c0 + p.chunk);
  const int nsub = c1 > c0 ? (c1 - c0 + kSub - 1) / kSub : 0;
  const bool resident = nsub <= 1;
  const T* __restrict__ xg = static_cast<const T*>(p.x);
  T* __restrict__ yg = static_cast<T*>(p.y);

  if (ncta > 1) cluster_sync();  // every CTA of the cluster runs before any DSMEM store

  auto load_sub = [&](const T* xr, int base, float* v, auto keep_l2) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int col0 = base + (k * kThreads + tid) * E;
      if (kVecIO && col0 < c1) {
        IO::template load_vec<decltype(keep_l2)::value>(xr + col0, v + k * E);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
          v[k * E + e] = (!kVecIO && col0 + e < c1) ? IO::load_one(xr + col0 + e) : -INFINITY;
      }
    }
  };
  auto store_sub = [&](T* yr, int base, const float* v) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int col0 = base + (k * kThreads + tid) * E;
      if (kVecIO) {
        if (col0 < c1) IO::store_vec(yr + col0, v + k * E);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (col0 + e < c1) IO::store_one(yr + col0 + e, v[k * E + e]);
      }
    }
  };

  float v[kPer];
  int it = 0;
  for (long long row = group; row < p.rows; row += groups, ++it) {
    const int par = it & 1;
    const T* xr = xg + row * p.cols;
    T* yr = yg + row * p.cols;

    // ---- pass 1: running (m, l) of this thread's slice
    float m = -INFINITY, l = 0.f, ref = 0.f;
    for (int sb = 0; sb < nsub; ++sb) {
      if (resident)
        load_sub(xr, c0, v, std::false_type{});
      else
        load_sub(xr, c0 + sb * kSub, v, std::true_type{});
      float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int i = 4; i < kPer; i += 4)
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], v[i + u]);
      const float gmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      if (gmax > m) {  // new running max: rescale the sum so far (l = 0 while m = -inf)
        l *= ex2_approx((m - gmax) * kLog2e);
        m = gmax;
      }
      ref = (m == -INFINITY) ? 0.f : m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const float e = ex2_approx((v[i] - ref) * kLog2e);
        acc[i & 3] += e;
        v[i] = e;  // kept for pass 2 when the slice is resident
      }
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }

    // ---- combine the threads' pairs (fixed order: every thread ends with the same values)
    const float2 bp = block_pair<kThreads>(m, l, warp_part, par);
    const float bm = bp.x, bl = bp.y;
    float M = bm, L = bl;
    if (ncta > 1) {
      // every CTA's pair goes to slot `rank` of every CTA; then each merges
      // the slots in rank order
      if (tid < ncta)
        st_shared_cluster_f32x2(mapa_shared(smem_u32(&peer_part[par][rank]), tid), bm, bl);
      cluster_sync();
      const float2 q0 = peer_part[par][0];
      M = q0.x;
      L = q0.y;
      for (int r = 1; r < ncta; ++r) {
        const float2 q = peer_part[par][r];
        merge_pair(M, L, q.x, q.y);
      }
    }
    if (rank == 0 && tid == 0 && p.lse) p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;

    // ---- pass 2: y = exp(x - M) / L
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float rM = (M == -INFINITY) ? 0.f : M;
    if (resident) {
      if (nsub == 1) {
        const float f = ex2_approx((ref - rM) * kLog2e) * inv;  // exp(ref_thread - M) / L
#pragma unroll
        for (int i = 0; i < kPer; ++i) v[i] *= f;
        store_sub(yr, c0, v);
      }
    } else {
      for (int sb = 0; sb < nsub; ++sb) {
        const int base = c0 + sb * kSub;
        load_sub(xr, base, v, std::true_type{});
#pragma unroll
        for (int i = 0; i < kPer; ++i) v[i] = ex2_approx((v[i] - rM) * kLog2e) * inv;
        store_sub(yr, base, v);
      }
    }
  }
  if (ncta > 1) cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// Rows with 16-byte aligned starts: the CTA's columns of each row come through
// a ring of kStages shared-memory stages (one sub-chunk of kThreads x 4
// vectors each), filled by bulk copies that thread 0 issues kStages items
// ahead.  Items, in order, per row: the nsub sub-chunks of pass 1, then (only
// when nsub > 1) the same sub-chunks again for pass 2.
template <typename T, int kThreads, int kStages>
__global__ void __launch_bounds__(kThreads) fa_softmax_ring_kernel(const SoftmaxParams p) {
  using IO = Io<T>;
  constexpr int E = IO::E;
  constexpr int kVec = 4;
  constexpr int kPer = kVec * E;
  constexpr int kSub = kThreads * kPer;
  constexpr uint32_t kStageBytes = kThreads * kVec * 16;
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t peer_full[2];  // the cluster's pairs of one row have landed
  __shared__ float2 warp_part[2][kWarps];
  __shared__ __align__(16) float4 peer_part[2][kMaxCluster];  // (m, l, failed) of every CTA
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int ncta = p.cluster;
  const int rank = ncta > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const long long groups = gridDim.x / ncta;
  const long long group = blockIdx.x / ncta;
  const int c0 = rank * p.chunk;
  const int c1 = min(p.cols, c0 + p.chunk);
  const int nsub = c1 > c0 ? (c1 - c0 + kSub - 1) / kSub : 0;
  const int per_row = nsub <= 1 ? nsub : 2 * nsub;
  const long long my_rows = group < p.rows ? (p.rows - 1 - group) / groups + 1 : 0;
  const long long total = my_rows * per_row;
  const T* __restrict__ xg = static_cast<const T*>(p.x);
  T* __restrict__ yg = static_cast<T*>(p.y);
  const uint32_t ring0 = smem_u32(ring);
  const uint32_t bar0 = smem_u32(&full[0]);
  const uint32_t peer_bar0 = smem_u32(&peer_full[0]);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init(peer_bar0, 1);
    mbar_init(peer_bar0 + 8, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (ncta > 1) cluster_sync();  // every CTA of the cluster runs before any DSMEM store
  const WaitCtx wc{&abort_flag, p.status, p.timeout_ns};

  // Thread 0: start the copy of item i (if it exists) into stage i % kStages.
  long long issued = 0;
  auto issue = [&](long long i) {
    if (i >= total) return;
    const long long r_local = i / per_row;
    const int k = static_cast<int>(i % per_row);
    const int sb = k % nsub;
    const long long row = group + r_local * groups;
    const int col = c0 + sb * kSub;
    const uint32_t bytes = static_cast<uint32_t>(min(kSub, c1 - col)) * sizeof(T);
    const int s = static_cast<int>(i % kStages);
    // pass 1 of a streamed row asks L2 to keep the data for pass 2's read
    const uint64_t pol = (nsub > 1 && k < nsub) ? l2_policy_evict_last() : l2_policy_evict_first();
    mbar_arrive_expect_tx(bar0 + 8 * s, bytes);
    bulk_load(ring0 + s * kStageBytes, xg + row * p.cols + col, bytes, bar0 + 8 * s, pol);
    issued = i + 1;
  };
  if (tid == 0)
    for (int i = 0; i < kStages; ++i) issue(i);

  long long q = 0;  // next item to consume
  bool failed = false;
  float v[kPer];
  // Wait for item q, copy this thread's vectors of it (columns from `base`,
  // -inf past c1), free the stage, start the copy kStages items ahead.
  // Returns false (block-uniform) once a wait has failed.
  auto consume = [&](int base) -> bool {
    const int s = static_cast<int>(q % kStages);
    const bool ok = !failed && wait_bounded(bar0 + 8 * s, static_cast<uint32_t>((q / kStages) & 1), wc);
    if (ok) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int slot = k * kThreads + tid;
        if (base + slot * E < c1) {
          uint32_t w[4];
          ld_shared_v4(ring0 + s * kStageBytes + slot * 16, w[0], w[1], w[2], w[3]);
          if constexpr (E == 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[k * 4 + e] = __uint_as_float(w[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[k * 8 + 2 * e] = __uint_as_float(w[e] << 16);
              v[k * 8 + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) v[k * E + e] = -INFINITY;
        }
      }
    }
    const bool bad = __syncthreads_or(!ok) != 0;
    if (!bad && tid == 0) issue(q + kStages);
    ++q;
    return !bad;
  };
  auto store = [&](T* yr, int base) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int col0 = base + (k * kThreads + tid) * E;
      if (col0 < c1) IO::store_vec(yr + col0, v + k * E);
    }
  };

  for (long long it = 0; it < my_rows; ++it) {
    const int par = static_cast<int>(it & 1);
    const long long row = group + it * groups;
    T* yr = yg + row * p.cols;

    // ---- pass 1
    float m = -INFINITY, l = 0.f, ref = 0.f;
    for (int sb = 0; sb < nsub; ++sb) {
      if (!consume(c0 + sb * kSub)) {
        failed = true;
        continue;
      }
      float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int i = 4; i < kPer; i += 4)
#pragma unroll
        for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], v[i + u]);
      const float gmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      if (gmax > m) {
        l *= ex2_approx((m - gmax) * kLog2e);
        m = gmax;
      }
      ref = (m == -INFINITY) ? 0.f : m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const float e = ex2_approx((v[i] - ref) * kLog2e);
        acc[i & 3] += e;
        v[i] = e;
      }
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }

    // ---- (M, L) of the row; a failed wait anywhere in the cluster stops every CTA here
    const float2 b = block_pair<kThreads>(m, l, warp_part, par);
    float M = b.x, L = b.y;
    bool any_failed = failed;
    if (ncta > 1) {
      // Send this CTA's pair to slot `rank` of every CTA (itself included)
      // with st.async, counted on the receiver's peer_full[par]; then wait
      // until all ncta pairs of this row have landed here.  A CTA sends row
      // `it` only after it has received every pair of row it-1, so no peer
      // still reads the slots of row it-2 that this overwrites.
      const uint32_t pb = peer_bar0 + 8 * par;
      if (tid == 0) mbar_arrive_expect_tx(pb, 16u * static_cast<uint32_t>(ncta));
      if (tid < ncta)
        st_async_f32x4(mapa_shared(smem_u32(&peer_part[par][rank]), tid), b.x, b.y,
                       failed ? 1.f : 0.f, 0.f, mapa_shared(pb, tid));
      const bool got = wait_bounded(pb, static_cast<uint32_t>((it >> 1) & 1), wc);
      if (__syncthreads_or(!got)) {
        failed = true;
        break;  // a peer never delivered: every CTA of the cluster times out here
      }
      const float4 q0 = peer_part[par][0];
      M = q0.x;
      L = q0.y;
      any_failed = q0.z != 0.f;
      for (int r = 1; r < ncta; ++r) {
        const float4 qr = peer_part[par][r];
        merge_pair(M, L, qr.x, qr.y);
        any_failed = any_failed || qr.z != 0.f;
      }
    }
    if (any_failed) break;
    if (rank == 0 && tid == 0 && p.lse) p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;

    // ---- pass 2: y = exp(x - M) / L
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float rM = (M == -INFINITY) ? 0.f : M;
    if (nsub == 1) {
      const float f = ex2_approx((ref - rM) * kLog2e) * inv;  // exp(ref_thread - M) / L
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] *= f;
      store(yr, c0);
    } else {
      for (int sb = 0; sb < nsub; ++sb) {
        if (!consume(c0 + sb * kSub)) {
          failed = true;  // reported at the next row's exchange
          continue;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) v[i] = ex2_approx((v[i] - rM) * kLog2e) * inv;
        store(yr, c0 + sb * kSub);
      }
    }
  }
  // copies still in flight (after a failure) land before the CTA may exit
  if (tid == 0)
    for (long long i = q; i < issued; ++i)
      wait_own(bar0 + 8 * static_cast<int>(i % kStages), static_cast<uint32_t>((i / kStages) & 1),
               p.timeout_ns);
  if (ncta > 1) cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// Persistent launch: as many CTAs (or clusters of p.cluster CTAs) as are
// resident at once, each looping over rows.  Clusters are co-scheduled inside
// one GPC, so their count comes from the occupancy query for that cluster
// shape, not from CTAs per SM x SMs (which would leave a second, nearly empty
// wave).
template <typename Kern>
cudaError_t launch_persistent(Kern kern, int threads, int smem, int per_sm,
                              std::atomic<int>* clusters_cache, const SoftmaxParams& p, int num_sms,
                              cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.cluster > 1 ? 1 : 0;
  long long slots = static_cast<long long>(per_sm) * num_sms;
  if (p.cluster > 1) {
    int clusters = clusters_cache[p.cluster].load(std::memory_order_relaxed);
    if (clusters == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(p.cluster));
      cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) clusters = 1;
      clusters_cache[p.cluster].store(clusters, std::memory_order_relaxed);
    }
    slots = clusters;
  }
  const long long groups = p.rows < slots ? p.rows : slots;
  cfg.gridDim = dim3(static_cast<unsigned>(groups * p.cluster));
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T, int kThreads>
cudaError_t launch_ring(const SoftmaxParams& p, int num_sms, cudaStream_t s) {
  constexpr int kStages = 3;  // 3 x 64 KB at 1024 threads
  constexpr int kSmem = kStages * kThreads * 64;
  auto kern = fa_softmax_ring_kernel<T, kThreads, kStages>;
  static std::atomic<int> cached{0};  // resident CTAs per SM (same on every sm_103 device)
  int per_sm = cached.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    cached.store(per_sm, std::memory_order_relaxed);
  }
  static std::atomic<int> clusters[kMaxCluster + 1] = {};
  return launch_persistent(kern, kThreads, kSmem, per_sm, clusters, p, num_sms, s);
}

template <typename T, int kThreads, bool kVecIO>
cudaError_t launch_one(const SoftmaxParams& p, int num_sms, cudaStream_t s) {
  auto kern = fa_softmax_rows_kernel<T, kThreads, 4, kVecIO>;
  static std::atomic<int> cached{0};  // resident CTAs per SM (same on every sm_103 device)
  int per_sm = cached.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    cached.store(per_sm, std::memory_order_relaxed);
  }
  static std::atomic<int> clusters[kMaxCluster + 1] = {};
  return launch_persistent(kern, kThreads, 0, per_sm, clusters, p, num_sms, s);
}

template <typename T, bool kVecIO>
cudaError_t launch_typed(SoftmaxParams p, int num_sms, cudaStream_t s) {
  constexpr int E = Io<T>::E;
  constexpr int kPer = 4 * E;
  // One CTA per row if the row fits in 32..1024 threads x kPer values: the
  // register kernel, several CTAs per SM overlapping each other's loads,
  // reductions and stores (measured faster than the ring at these sizes).
  for (int t = 32; t <= 1024; t *= 2) {
    if (p.cols <= t * kPer) {
      p.cluster = 1;
      p.chunk = t * kPer;
      switch (t) {
        case 32: return launch_one<T, 32, kVecIO>(p, num_sms, s);
        case 64: return launch_one<T, 64, kVecIO>(p, num_sms, s);
        case 128: return launch_one<T, 128, kVecIO>(p, num_sms, s);
        case 256: return launch_one<T, 256, kVecIO>(p, num_sms, s);
        case 512: return launch_one<T, 512, kVecIO>(p, num_sms, s);
        default: return launch_one<T, 1024, kVecIO>(p, num_sms, s);
      }
    }
  }
  // A cluster of CTAs of 1024 threads shares the row in equal chunks (whole
  // 16-byte vectors): resident up to 8 CTAs, beyond that 8 CTAs stream
  // sub-chunks of their chunk.
  constexpr int kCap = 1024 * kPer;
  const long long need = (static_cast<long long>(p.cols) + kCap - 1) / kCap;
  p.cluster = static_cast<int>(need < kMaxCluster ? need : kMaxCluster);
  const long long per = (static_cast<long long>(p.cols) + p.cluster - 1) / p.cluster;
  p.chunk = static_cast<int>((per + E - 1) / E * E);
  if (kVecIO) return launch_ring<T, 1024>(p, num_sms, s);
  return launch_one<T, 1024, false>(p, num_sms, s);
}

}  // namespace

cudaError_t launch_softmax_rows(const SoftmaxParams& p, bool bf16, bool vec_io, int num_sms,
                                cudaStream_t s) {
  if (bf16)
    return vec_io ? launch_typed<__nv_bfloat16, true>(p, num_sms, s)
                  : launch_typed<__nv_bfloat16, false>(p, num_sms, s);
  return vec_io ? launch_typed<float, true>(p, num_sms, s) : launch_typed<float, false>(p, num_sms, s);
}

}  // namespace fa
