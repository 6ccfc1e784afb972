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
// registers, several CTAs per SM overlapping one another, the row read from
// HBM once; pass 2 rescales the exponentials kept from pass 1 by
// exp(m_thread - M) / L.  Longer rows with 16-byte aligned starts, when there
// are at least two per SM, run fa_softmax_stream_kernel: one CTA per row at a
// time (two per SM), the row streamed through a shared-memory ring of 1-D bulk
// copies (TMA) twice, the second time from L2, and no CTA ever waits for
// another.  Fewer long rows run fa_softmax_ring_kernel on a cluster of up to 8
// CTAs of 1024 threads that share the row: each CTA's columns arrive through
// its own ring; a row that fits the cluster's registers is read once, longer
// rows are cut into sub-chunks that pass 2 streams through the ring again.
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
constexpr int kMaxStreamGroup = 16;  // a non-portable cluster size, allowed per kernel
// The streaming kernel runs two CTAs per SM; a group of CTAs shares each
// row, and long rows stream that way when there is at least one row per
// group.  Fewer rows share each row across a cluster of the ring kernel.
constexpr long long kStreamCtasPerSm = 2;
// The streaming kernel asks L2 for the next row's first sub-chunk only while
// the rows in flight (one per group) take at most this much of L2.
constexpr long long kStreamPrefetchL2Bytes = 96ll << 20;

// CTAs per row for the streaming kernel: the group sizes that measured
// fastest on GB300 for rows of 32K-4M elements.  Longer chunks per CTA keep
// more rows in flight (more L2 misses between the passes, longer pipeline
// fill per row); more CTAs per row pay more exchanges and smaller loads.
template <typename T>
int stream_group(long long cols) {
  if (sizeof(T) == 4) {
    if (cols <= 20480) return 1;
    if (cols <= 40960) return 2;
    if (cols <= 131072) return 4;
    if (cols <= 524288) return 8;
    return 16;
  }
  if (cols <= 65536) return 1;
  if (cols <= 262144) return 2;
  if (cols <= 524288) return 4;
  return 8;  // 16 measured slower for bf16 rows of 2M
}

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

// Shared-memory add with acquire-release order at CTA scope; returns the old
// value.  The caller's earlier shared-memory accesses happen before it, and
// whatever the caller does next happens after every earlier add to `addr`.
__device__ __forceinline__ uint32_t atom_add_acq_rel_smem(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

// Global -> L2 only (no shared memory, no completion signal), `bytes` a
// multiple of 16 from a 16-byte aligned address.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
               "r"(bytes), "l"(policy)
               : "memory");
}

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

// Largest of v[0..N) with three-input max instructions (N a multiple of 4):
// four running maxima, each taking two new values per step.
template <int N>
__device__ __forceinline__ float max_of(const float* v) {
  float mx[4] = {v[0], v[1], v[2], v[3]};
  int i = 4;
#pragma unroll
  for (; i + 8 <= N; i += 8)
#pragma unroll
    for (int u = 0; u < 4; ++u) mx[u] = max3f(mx[u], v[i + u], v[i + 4 + u]);
#pragma unroll
  for (; i < N; i += 4)
#pragma unroll
    for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], v[i + u]);
  return fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
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

// Long rows, at least one per resident CTA group: a group of kCta CTAs (a
// cluster when kCta > 1) takes one row at a time, each CTA streaming its
// chunk of the row through a ring of kStages shared-memory stages filled by
// 1-D bulk copies -- pass 1 from HBM (the copies ask L2 to keep the lines),
// pass 2 again from L2 -- so every group works on its own rows and L2 holds
// about one row per group between the passes.  Pass 1 ends on the chunk's
// last sub-chunk, whose exponentials are still in registers: pass 2 writes
// that sub-chunk first, from the registers, and reloads only the other
// nsub - 1 (so pass 1 marks the last one evict-first).  Loads of a row, in
// order: sub-chunks 0 .. nsub-1 (pass 1), then 0 .. nsub-2 (pass 2).
//
// The warps never meet at a CTA-wide barrier.  Each waits for a stage on its
// own, copies its vectors to registers and counts itself out of the stage; the
// warp that counts the stage empty starts the load kStages ahead into it
// (stages are released in load order, so load g lives in stage g % kStages).
// At the end of pass 1 every warp publishes its (m, l) and arrives on the
// row's mbarrier; each warp then merges all warps' pairs itself (the same tree
// in every warp) while the ring keeps loading.  In a cluster, warp 0 of each
// CTA then sends the CTA's pair to every CTA of the group (st.async, counted
// on the receiver's mbarrier) and every warp merges the group's pairs in rank
// order, so all CTAs of a row get the same (M, L).
template <typename T, int kWarps, int kVec, int kStages, int kCta>
__global__ void __launch_bounds__(kWarps * 32, 1024 / (kWarps * 32))
    fa_softmax_stream_kernel(const SoftmaxParams p) {
  using IO = Io<T>;
  constexpr int kThreads = kWarps * 32;
  constexpr int E = IO::E;
  constexpr int kPer = kVec * E;
  constexpr int kSub = kThreads * kPer;  // columns per sub-chunk
  constexpr uint32_t kStageBytes = kThreads * kVec * 16;
  // Pair slots and their mbarriers cycle over 4 rows.  A warp publishes row
  // it+4 after its wait for the last pass-1 load of that row, started only
  // once every warp had released the load kStages earlier -- one of row it+1
  // or later, as rows hold per_row = 2 * nsub - 1 loads and
  // 3 * per_row + nsub - 1 >= 3 >= kStages -- and every warp reads the pairs
  // of row it before releasing any load of row it+1.  A peer CTA sends its
  // pair of row it+4 only after receiving ours of row it+3, which we send
  // after every warp here has finished with row it.
  constexpr int kSlots = 4;
  static_assert(kStages >= 2 && kStages <= 3, "ring depth");
  static_assert(kCta >= 1 && kCta <= kMaxStreamGroup, "group size");
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t red[kSlots];        // all warps' pairs of a row are published
  __shared__ __align__(8) uint64_t peer_full[kSlots];  // all CTAs' pairs of a row have landed
  __shared__ uint32_t reads[kStages];                  // warp releases of the stage, ever
  __shared__ float2 warp_part[kSlots][kWarps];
  __shared__ __align__(16) float4 peer_part[kSlots][kCta];  // (m, l, failed, -) per CTA
  __shared__ long long issued_sh;  // loads whose copies have been started
  __shared__ int abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = kCta > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const long long groups = gridDim.x / kCta;
  const long long group = blockIdx.x / kCta;
  const int c0 = rank * p.chunk;  // this CTA's columns [c0, c1) of every row
  const int c1 = min(p.cols, c0 + p.chunk);
  const int nsub = c1 > c0 ? (c1 - c0 + kSub - 1) / kSub : 0;
  const int per_row = nsub > 0 ? 2 * nsub - 1 : 0;  // loads per row
  const long long my_rows = group < p.rows ? (p.rows - 1 - group) / groups + 1 : 0;
  const long long total = my_rows * per_row;
  const bool pf_ok = groups * p.cols * static_cast<long long>(sizeof(T)) <= kStreamPrefetchL2Bytes;
  const T* __restrict__ xg = static_cast<const T*>(p.x);
  T* __restrict__ yg = static_cast<T*>(p.y);
  const uint32_t ring0 = smem_u32(ring);
  const uint32_t bar0 = smem_u32(&full[0]);
  const uint32_t red0 = smem_u32(&red[0]);
  const uint32_t peer0 = smem_u32(&peer_full[0]);
  const uint32_t reads0 = smem_u32(&reads[0]);

  // Start load g (if it exists) into stage g % kStages.
  auto issue = [&](long long g) {
    if (g >= total) return;
    const long long row = group + (g / per_row) * groups;
    const int k = static_cast<int>(g % per_row);
    const int col = c0 + (k < nsub ? k : k - nsub) * kSub;
    const uint32_t bytes = static_cast<uint32_t>(min(kSub, c1 - col)) * sizeof(T);
    const int s = static_cast<int>(g % kStages);
    // pass-1 loads that pass 2 reads again ask L2 to keep them
    const uint64_t pol = k < nsub - 1 ? l2_policy_evict_last() : l2_policy_evict_first();
    if (FA_DCHECK(row < p.rows && col < c1, p.status)) {
      mbar_arrive_expect_tx(bar0 + 8 * s, bytes);
      bulk_load(ring0 + s * kStageBytes, xg + row * p.cols + col, bytes, bar0 + 8 * s, pol);
    }
    *reinterpret_cast<volatile long long*>(&issued_sh) = g + 1;
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar0 + 8 * s, 1);
      reads[s] = 0;
    }
    for (int r = 0; r < kSlots; ++r) {
      mbar_init(red0 + 8 * r, kWarps);
      mbar_init(peer0 + 8 * r, 1);
    }
    abort_flag = 0;
    issued_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (kCta > 1) cluster_sync();  // every CTA of the group runs before any DSMEM store
  if (tid == 0)
    for (int g = 0; g < kStages; ++g) issue(g);
  const WaitCtx wc{&abort_flag, p.status, p.timeout_ns};

  long long g = 0;  // next load this warp uses
  float v[kPer];
  // Wait for load g, copy this thread's vectors of it (columns from `base`,
  // -inf past the chunk's end), count the warp out of the stage (the last
  // warp out refills it).  False (warp-uniform) if the wait failed.
  auto take = [&](int base) -> bool {
    const int s = static_cast<int>(g % kStages);
    if (!warp_wait(bar0 + 8 * s, static_cast<uint32_t>((g / kStages) & 1), wc)) return false;
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
    __syncwarp();
    if (lane == 0) {
      const uint32_t before = atom_add_acq_rel_smem(reads0 + 4 * s, 1);
      if ((before + 1) % kWarps == 0) {
        fence_proxy_async_smem();
        issue(g + kStages);
      }
    }
    ++g;
    return true;
  };
  auto store = [&](T* yr, int base) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int col0 = base + (k * kThreads + tid) * E;
      if (col0 < c1) IO::store_vec(yr + col0, v + k * E);
    }
  };

  const uint64_t l2e = f2_pack(kLog2e, kLog2e);
  bool failed = false;
  for (long long it = 0; it < my_rows && !failed; ++it) {
    const long long row = group + it * groups;
    T* yr = yg + row * p.cols;
    const int slot = static_cast<int>(it % kSlots);
    const uint32_t slot_par = static_cast<uint32_t>((it / kSlots) & 1);
    // this CTA expects every group member's pair of the row (its own included)
    if (kCta > 1 && tid == 0) mbar_arrive_expect_tx(peer0 + 8 * slot, 16u * kCta);

    // ---- pass 1: running (m, l) of this thread's columns; v keeps the last
    // sub-chunk's exponentials, taken against `ref`
    float m = -INFINITY, l = 0.f, ref = 0.f;
    for (int sc = 0; sc < nsub; ++sc) {
      if (!take(c0 + sc * kSub)) {
        failed = true;
        break;
      }
      const float gmax = max_of<kPer>(v);
      if (gmax > m) {  // new running max: rescale the sum so far (l = 0 while m = -inf)
        l *= ex2_approx((m - gmax) * kLog2e);
        m = gmax;
      }
      ref = (m == -INFINITY) ? 0.f : m;
      const uint64_t nref = f2_pack(-ref, -ref);
      uint64_t acc[2] = {0, 0};
#pragma unroll
      for (int i = 0; i < kPer; i += 2) {
        float a, b;
        f2_unpack(fmul2(fadd2(f2_pack(v[i], v[i + 1]), nref), l2e), a, b);
        const uint64_t e = f2_pack(ex2_approx(a), ex2_approx(b));
        acc[(i >> 1) & 1] = fadd2(acc[(i >> 1) & 1], e);
        f2_unpack(e, v[i], v[i + 1]);
      }
      float a0, a1, a2, a3;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], a2, a3);
      l += (a0 + a1) + (a2 + a3);
    }
    // a failed CTA still publishes (flagged) so that its group does not wait
    // for it until the limit

    // ---- (M, L) of the CTA's chunk from every warp's pair
    const float2 wp = warp_pair(m, l);
    if (lane == 0) {
      warp_part[slot][warp] = wp;
      mbar_arrive(red0 + 8 * slot);  // release: the pair is written before the arrival
    }
    if (!warp_wait(red0 + 8 * slot, slot_par, wc)) failed = true;
    const float2 bp = lane < kWarps ? warp_part[slot][lane] : make_float2(-INFINITY, 0.f);
    float2 ML = warp_pair(bp.x, bp.y);
    if (kCta > 1) {
      // ---- the group's pairs, merged in rank order
      if (warp == 0 && lane < kCta)
        st_async_f32x4(mapa_shared(smem_u32(&peer_part[slot][rank]), lane), ML.x, ML.y,
                       failed ? 1.f : 0.f, 0.f, mapa_shared(peer0 + 8 * slot, lane));
      if (!warp_wait(peer0 + 8 * slot, slot_par, wc)) {
        failed = true;
        break;
      }
      const float4 q0 = peer_part[slot][0];
      ML = make_float2(q0.x, q0.y);
      bool any_failed = q0.z != 0.f;
#pragma unroll
      for (int r = 1; r < kCta; ++r) {
        const float4 qr = peer_part[slot][r];
        merge_pair(ML.x, ML.y, qr.x, qr.y);
        any_failed = any_failed || qr.z != 0.f;
      }
      if (any_failed) failed = true;
    }
    if (failed) break;
    const float M = ML.x, L = ML.y;
    if (rank == 0 && warp == 0 && lane == 0 && p.lse)
      p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;

    // ---- pass 2: y = exp(x - M) / L, the last sub-chunk from the registers
    // (exp(x - ref) * exp(ref - M) / L), the others reloaded
    // While this CTA re-reads the row from L2, ask L2 for the first sub-chunk
    // of its next row, so HBM stays busy and that row's first load hits L2 --
    // unless the rows in flight already overflow L2 (one per group), or the
    // chunk has fewer than three sub-chunks (measured slower either way).
    if (warp == 0 && lane == 0 && it + 1 < my_rows && nsub >= 3 && pf_ok) {
      const long long nrow = row + groups;
      for (int sc = 0; sc < 1 && sc < nsub; ++sc) {
        const int col = c0 + sc * kSub;
        const uint32_t bytes = static_cast<uint32_t>(min(kSub, c1 - col)) * sizeof(T);
        bulk_prefetch_l2(xg + nrow * p.cols + col, bytes,
                         sc < nsub - 1 ? l2_policy_evict_last() : l2_policy_evict_first());
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float rM = (M == -INFINITY) ? 0.f : M;
    if (nsub > 0) {
      const float f = ex2_approx((ref - rM) * kLog2e) * inv;
      const uint64_t f2 = f2_pack(f, f);
#pragma unroll
      for (int i = 0; i < kPer; i += 2)
        f2_unpack(fmul2(f2_pack(v[i], v[i + 1]), f2), v[i], v[i + 1]);
      store(yr, c0 + (nsub - 1) * kSub);
    }
    // the reloaded sub-chunks: y = 2^((x - M) log2 e - log2 L), the division
    // folded into the exponent.  L >= 1 (the row max contributes 1), so
    // log2 L = e + log2 f with L = 2^e f, f in [1, 2): the exponent field plus
    // lg2.approx on f (absolute error about 2^-22), and the rounded sum adds at
    // most 2^-19 (|log2 L| <= 31) to the exponent's error.
    float nl2L = -INFINITY;
    if (L > 0.f) {
      const uint32_t bits = __float_as_uint(L);
      const float f = __uint_as_float((bits & 0x007FFFFFu) | 0x3F800000u);
      nl2L = -(static_cast<float>(static_cast<int>(bits >> 23) - 127) + __log2f(f));
    }
    const uint64_t nrM = f2_pack(-rM, -rM), nl2 = f2_pack(nl2L, nl2L);
    for (int sc = 0; sc + 1 < nsub; ++sc) {
      if (!take(c0 + sc * kSub)) {
        failed = true;
        break;
      }
#pragma unroll
      for (int i = 0; i < kPer; i += 2) {
        float a, c;
        f2_unpack(ffma2(fadd2(f2_pack(v[i], v[i + 1]), nrM), l2e, nl2), a, c);
        v[i] = ex2_approx(a);
        v[i + 1] = ex2_approx(c);
      }
      store(yr, c0 + sc * kSub);
    }
  }
  // Copies still in flight (after a failure) land before the CTA may exit:
  // each stage's latest copy is one of the last kStages issued.
  __syncthreads();
  if (tid == 0) {
    const long long issued = issued_sh;
    for (long long i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
      wait_own(bar0 + 8 * static_cast<int>(i % kStages), static_cast<uint32_t>((i / kStages) & 1),
               p.timeout_ns);
  }
  if (kCta > 1) cluster_sync();  // no CTA leaves while a peer may still address its shared memory
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

template <typename T, int kWarps, int kVec, int kStages, int kCta>
cudaError_t launch_stream(const SoftmaxParams& p, int num_sms, cudaStream_t s) {
  constexpr int kSmem = kStages * kWarps * 32 * kVec * 16;
  auto kern = fa_softmax_stream_kernel<T, kWarps, kVec, kStages, kCta>;
  static std::atomic<int> cached{0};  // resident CTAs per SM (same on every sm_103 device)
  int per_sm = cached.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (kCta > kMaxCluster) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, kSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    cached.store(per_sm, std::memory_order_relaxed);
  }
  static std::atomic<int> clusters[kCta + 1] = {};
  return launch_persistent(kern, kWarps * 32, kSmem, per_sm, clusters, p, num_sms, s);
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
  // Long rows, at least one per group of CTAs: each group (a cluster of
  // stream_group CTAs) takes one row at a time and streams it twice (the
  // second time mostly from L2).
  if (kVecIO) {
    const int cta = stream_group<T>(p.cols);
    if (p.rows * cta >= kStreamCtasPerSm * static_cast<long long>(num_sms)) {
      p.cluster = cta;
      p.chunk = static_cast<int>((static_cast<long long>(p.cols) + cta * E - 1) / (cta * E) * E);
      switch (cta) {
        case 1: return launch_stream<T, 16, 4, 3, 1>(p, num_sms, s);
        case 2: return launch_stream<T, 16, 4, 3, 2>(p, num_sms, s);
        case 4: return launch_stream<T, 16, 4, 3, 4>(p, num_sms, s);
        case 8: return launch_stream<T, 16, 4, 3, 8>(p, num_sms, s);
        default: return launch_stream<T, 16, 4, 3, 16>(p, num_sms, s);
      }
    }
  }
  // Otherwise a cluster of CTAs of 1024 threads shares the row in equal
  // chunks (whole 16-byte vectors): resident up to 8 CTAs, beyond that 8 CTAs
  // stream sub-chunks of their chunk.
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
