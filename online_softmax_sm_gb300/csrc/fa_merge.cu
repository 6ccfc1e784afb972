// fa_merge.cu -- combine n_splits partial (m, l, O) triples per query row.
//
// The two-block merge rule (airsota.com online-softmax card, section 三,
// "Running Combined Updates"), written in its n-way form, which the rule's
// associativity ("La recurrencia del online softmax", practice problem 4)
// makes equal to any sequence of pairwise merges:
//   M   = max_s m_s
//   w_s = l_s exp(m_s - M)      (0 for an empty split, m_s = -inf)
//   l   = sum_s w_s
//   O   = sum_s w_s O_s / l      (O_s already normalised by l_s)
//   LSE = M + ln l;  a row with l = 0 gets O = 0 and LSE = -inf.
// m_s is in natural-log units of the scaled logits.  HBM-bound: each row reads
// n_splits * (d + 2) fp32 (or n_splits * (2 fp32 + d bf16) when fa_fwd's own
// workspace holds O_s in bf16) and writes d bf16 + one fp32.  d/8 lanes own a
// row, eight consecutive columns each: two 16-byte loads per split (one for
// bf16; four splits' loads in flight at once), one 16-byte store of bf16 O.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {

template <int D, bool kBf16Part>
__global__ void __launch_bounds__(256) fa_merge_kernel(const MergeParams p) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kU = 4;  // splits whose loads are in flight together
  const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = g / kLanesPerRow;
  const int part = static_cast<int>(g % kLanesPerRow);
  if (row >= p.rows) return;
  const int S = p.n_splits;

  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, __ldg(p.m_part + s * p.rows + row));

  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  float lsum = 0.f;
  // this lane's eight columns of split row idx: two 16-byte fp32 loads, or
  // one 16-byte load of bf16 (exact in fp32)
  auto load_o = [&](long long idx, float4& a, float4& b) {
    if constexpr (kBf16Part) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(p.o_part) + idx * D + part * 8));
      a = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                      __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      b = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u),
                      __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
    } else {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.o_part) + idx * D + part * 8);
      a = __ldg(src);
      b = __ldg(src + 1);
    }
  };
  // Splits in ascending order, as one sequence of FMAs; groups of kU splits
  // issue all their loads before the first use, so each thread keeps 2 * kU
  // 16-byte loads in flight instead of two.
  auto fold = [&](float ms, float ls, const float4& a, const float4& b) {
    if (ms == -INFINITY) return;  // an empty split adds nothing
    const float w = ls * expf(ms - M);
    lsum += w;
    acc[0] = fmaf(w, a.x, acc[0]);
    acc[1] = fmaf(w, a.y, acc[1]);
    acc[2] = fmaf(w, a.z, acc[2]);
    acc[3] = fmaf(w, a.w, acc[3]);
    acc[4] = fmaf(w, b.x, acc[4]);
    acc[5] = fmaf(w, b.y, acc[5]);
    acc[6] = fmaf(w, b.z, acc[6]);
    acc[7] = fmaf(w, b.w, acc[7]);
  };
  if (M != -INFINITY) {
    int s = 0;
    for (; s + kU <= S; s += kU) {
      float ms[kU], ls[kU];
      float4 a[kU], b[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const long long idx = static_cast<long long>(s + u) * p.rows + row;
        ms[u] = __ldg(p.m_part + idx);
        ls[u] = __ldg(p.l_part + idx);
        load_o(idx, a[u], b[u]);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) fold(ms[u], ls[u], a[u], b[u]);
    }
    for (; s < S; ++s) {
      const long long idx = static_cast<long long>(s) * p.rows + row;
      float4 a, b;
      load_o(idx, a, b);
      fold(__ldg(p.m_part + idx), __ldg(p.l_part + idx), a, b);
    }
  }
  const bool empty = !(lsum > 0.f);
  const float inv = empty ? 0.f : 1.f / lsum;
  uint4 out;
  __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[4] * inv, acc[5] * inv);
  __nv_bfloat162 h3 = __floats2bfloat162_rn(acc[6] * inv, acc[7] * inv);
  out.x = *reinterpret_cast<uint32_t*>(&h0);
  out.y = *reinterpret_cast<uint32_t*>(&h1);
  out.z = *reinterpret_cast<uint32_t*>(&h2);
  out.w = *reinterpret_cast<uint32_t*>(&h3);
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + row * D + part * 8) = out;
  if (part == 0) p.lse[row] = empty ? -INFINITY : M + logf(lsum);
}

cudaError_t launch_merge(int d, const MergeParams& p, cudaStream_t s) {
  const long long threads = p.rows * (d / 8);
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (blocks == 0) return cudaSuccess;
  if (d == 64) {
    if (p.o_part_bf16)
      fa_merge_kernel<64, true><<<blocks, 256, 0, s>>>(p);
    else
      fa_merge_kernel<64, false><<<blocks, 256, 0, s>>>(p);
  } else {
    if (p.o_part_bf16)
      fa_merge_kernel<128, true><<<blocks, 256, 0, s>>>(p);
    else
      fa_merge_kernel<128, false><<<blocks, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa
