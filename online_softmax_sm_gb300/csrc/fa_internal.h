// fa_internal.h -- declarations shared by the library's translation units
// (kernel parameters, launcher prototypes, device status codes).  Not part of
// the public C ABI (that is include/fa.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Device status word values (written by kernels, read by fa_get_device_status).
enum : int {
  kDevOk = 0,
  kDevTimeout = 1,  // a bounded mbarrier wait ran out; the CTA stopped cleanly
  kDevCheck = 2,    // debug build (FA_DEBUG): a bounds check failed; the access was skipped
};
// The status word is the first of two ints per device; the second holds the
// source line of the first failed debug-build check.

// Default K/V tile (keys per tile): split-KV ranges are counted in these.
constexpr int kDefaultBc = 128;

// Division of 0 <= n < 2^31 by a divisor fixed at launch, as a multiply-high
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): q = (mulhi(n, mul) + n) >> shift.
struct FastDiv {
  unsigned int mul;
  unsigned int shift;
  int d;
};

inline FastDiv make_fastdiv(int d) {
  FastDiv f{0u, 0u, d};
  unsigned int s = 0;
  while ((1ull << s) < static_cast<unsigned long long>(d)) ++s;  // s = ceil(log2 d)
  f.shift = s;
  f.mul = static_cast<unsigned int>(((1ull << 32) * ((1ull << s) - static_cast<unsigned long long>(d))) /
                                        static_cast<unsigned long long>(d) + 1ull);
  return f;
}

struct FwdParams {
  // n_splits == 1: final outputs.  o is written by TMA through the O map (rows
  // with no visible key are zeroed through this pointer).
  void* o;     // bf16 [B*H][Nq][d]
  float* lse;  // [B*H][Nq]
  // partial != 0: write partial triples instead, index ((split * BH + bh) * Nq + row).
  int partial;
  float* m_part;  // natural-log units (scale * raw max), -inf if empty
  float* l_part;  // sum of exp(scale*s - m_part)
  void* o_part;   // [.., d] O_split / l_split (0 if empty): fp32, or bf16 if part_bf16
  int part_bf16;
  int Nq, Nk, BH;
  int n_splits;
  int tiles_per_split;  // K/V tiles per split
  int kv_tiles;         // ceil(Nk / BC)
  // Work items of one launch of the persistent grid: (query-tile group, split,
  // head) for heads [bh0, bh0 + n_bh) and splits [split0, split0 + n_split);
  // the host keeps n_items below 2^31 by cutting a launch into several.
  int n_items;          // n_qg * n_split * n_bh
  int rounds;           // ceil(n_items / grid size)
  int n_qg;             // groups of QT query tiles per head
  int bh0, n_bh;
  int split0, n_split;
  // qg_major: heads go in blocks of hb; within a block, item index =
  // (group, head, split).  Otherwise item index = (head, split, group).
  int qg_major;
  int hb;               // heads per block (qg_major)
  FastDiv div_qg, div_split;  // by n_qg, n_split
  FastDiv div_blk;            // by n_qg * n_split * hb (items of a full block)
  FastDiv div_per, div_per_last;  // by n_split * hb, and by n_split * (heads of the last block)
  int qg_desc;          // 1: groups in descending order (later groups see more keys)
  int wl, wr;        // visible keys [r + off - wl, r + off + wr]; -1 = open side
  float scale;       // natural-units logit scale
  float scale_log2;  // scale * log2(e)
  float o_scale;     // FP8 forward: final_scale = v_descale 2^-8 applied to O
  unsigned long long timeout_ns;
  int test_skip_load;  // >= 0: the producer skips this K/V load (test hook)
  int* status;         // device status word
};

struct MergeParams {
  const float* m_part;
  const float* l_part;
  const void* o_part;  // fp32, or bf16 if o_part_bf16
  int o_part_bf16;
  void* o;     // bf16 [rows][d]
  float* lse;  // [rows]
  long long rows;  // B*H*Nq
  int n_splits;
};

// Launchers (one per translation unit); return cudaSuccess or the launch error.
// qt: Q tiles (128 rows each) per CTA.
cudaError_t launch_fwd_d64_bc64(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                cudaStream_t s);
cudaError_t launch_fwd_d64_bc128(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                 cudaStream_t s);
cudaError_t launch_fwd_d128_bc64(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                 cudaStream_t s);
cudaError_t launch_fwd_d128_bc128(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                  cudaStream_t s);
cudaError_t launch_fwd_fp8_d128(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                cudaStream_t s);
cudaError_t launch_merge(int d, const MergeParams& p, cudaStream_t s);

// fa_fwd with n_splits > 1 and its split workspace in the caller's device
// memory (fa_api.cu; used by the no-alloc entry point): same kernels and
// layout as fa_fwd, so the same bits.
int fwd_split_into(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Nq, int Nk, int d, float scale, int causal, int n_splits, void* stream,
                   void* ws, size_t ws_bytes);

// Attention backward (fa_bwd_kernel.cuh).
struct BwdParams {
  int Nq, Nk, BH;
  int nq_pad;         // rows of nlse2 / nd per head (Nq rounded up to 128)
  int wl, wr;         // mask window, as FwdParams (causal = (-1, 0))
  int causal;         // launch order only
  float scale;        // natural-units logit scale
  float scale_log2;   // scale * log2(e)
  const float* nlse2; // [BH][nq_pad]: -LSE * log2(e); -inf where P must be 0
  const float* nd;    // [BH][nq_pad]: -D_i = -<dO_i, O_i>
  unsigned long long timeout_ns;
  int* status;
};

struct BwdPreParams {
  const void* o;      // bf16 [BH][Nq][d]
  const void* dout;   // bf16 [BH][Nq][d]
  const float* lse;   // [BH][Nq]
  float* nlse2;       // [BH][nq_pad]
  float* nd;          // [BH][nq_pad]
  int Nq, nq_pad, BH;
};

cudaError_t launch_bwd_d64(const CUtensorMap* maps, const BwdParams& p, const BwdPreParams& pre,
                           cudaStream_t s);
cudaError_t launch_bwd_d128(const CUtensorMap* maps, const BwdParams& p, const BwdPreParams& pre,
                            cudaStream_t s);

// Row softmax (fa_softmax.cu).  Row r's columns are split over `cluster`
// CTAs, `chunk` columns each (a multiple of the 16-byte vector width).
struct SoftmaxParams {
  const void* x;
  void* y;
  float* lse;  // may be null
  long long rows;
  int cols;
  int cluster;
  int chunk;
  int* status;                    // device status word (timed-out waits)
  unsigned long long timeout_ns;  // bound of each wait
};

cudaError_t launch_softmax_rows(const SoftmaxParams& p, bool bf16, bool vec_io, int num_sms,
                                cudaStream_t s);

}  // namespace fa
