// fa_api.cu -- the C ABI (include/fa.h): argument validation, TMA tensor
// maps, launch configuration, the split-KV workspace and error reporting.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"
#include "fa_status.h"

namespace {

constexpr int kVersion = 101;
constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait
constexpr int kMaxDevices = 64;
constexpr int kMaxSeq = 1 << 30;

thread_local cudaError_t t_last_cuda = cudaSuccess;
thread_local char t_msg[256];
thread_local char t_check_msg[160] = "debug build: a device-side bounds check failed";

// Device status words, one pair per device: [0] what went wrong (kernels
// record timed-out waits, and failed debug-build checks, here), [1] the
// source line of the first failed check.
__device__ int g_fa_status[2];

struct DevState {
  bool checked = false;
  bool supported = false;
  int* status = nullptr;
  int num_sms = 0;
};
DevState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int cuda_fail(cudaError_t e) {
  t_last_cuda = e;
  return FA_ERR_CUDA;
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Current device: sm_103 check and the status-word address, once per device.
int device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      if ((e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
          cudaSuccess)
        return cuda_fail(e);
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_fa_status)) != cudaSuccess) return cuda_fail(e);
      st.status = static_cast<int*>(p);
    }
    st.checked = true;
  }
  if (!st.supported) return FA_ERR_UNSUPPORTED;
  *out = &st;
  return FA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 3-D bf16 map over [batch][rows][inner] with a (64 x box_rows x 1) box and
// the 128-byte swizzle; out-of-range rows read as zero / are clipped on store.
int make_map(CUtensorMap* m, const void* base, int inner, int rows, int batch, int box_rows,
             bool bytes = false) {
  // bf16 elements (box 64 wide) or one-byte FP8 elements (box 128 wide): one
  // 128-byte swizzle row either way
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t es = bytes ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * es,
                                 static_cast<cuuint64_t>(inner) * es * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {bytes ? 128u : 64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

int check_sizes(int B, int H, int Nq, int Nk, int d, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (Nq > kMaxSeq || Nk > kMaxSeq) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

cudaError_t launch_fwd(int d, int bc, int qt, const CUtensorMap* maps, const fa::FwdParams& p,
                       dim3 grid, cudaStream_t s) {
  if (d == 64) return bc == 64 ? fa::launch_fwd_d64_bc64(qt, maps, p, grid, s)
                               : fa::launch_fwd_d64_bc128(qt, maps, p, grid, s);
  return bc == 64 ? fa::launch_fwd_d128_bc64(qt, maps, p, grid, s)
                  : fa::launch_fwd_d128_bc128(qt, maps, p, grid, s);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// K/V tiles item (query-tile group qg, whole key axis) streams: the host's
// copy of the kernel's per-item range (make_item), for scheduling only.
int item_steps(const fa::FwdParams& p, int qt, int qg, int bc) {
  const int off = p.Nk - p.Nq;
  int b = p.kv_tiles, e = 0;
  for (int i = 0; i < qt; ++i) {
    const int r_first = qg * 128 * qt + 128 * i;
    if (r_first >= p.Nq) continue;
    const int r_last = std::min(r_first + 128, p.Nq) - 1;
    const int klo = p.wl < 0 ? 0 : std::max(0, r_first + off - p.wl);
    const int khi = p.wr < 0 ? p.Nk - 1 : std::min(p.Nk - 1, r_last + off + p.wr);
    if (khi < klo) continue;
    b = std::min(b, klo / bc);
    e = std::max(e, khi / bc + 1);
  }
  return e > b ? e - b : 0;
}

// Heads per block of the masked order.  A mask makes the query-tile groups'
// work unequal; the snake deal evens out the CTAs' totals only for some block
// sizes, and larger blocks keep more heads' K/V live in L2 at once.  The
// balance of each candidate (powers of two, and all heads) is simulated on the
// host (the deal is static); among the candidates within 3 % of the best
// balance, the largest whose K/V fits in 64 MB wins, else the best-balanced.
int choose_heads_blk(const fa::FwdParams& p, int qt, int bc, int G, long long kv_head) {
  const int nb = p.n_bh;
  const long long items = static_cast<long long>(p.n_qg) * p.n_split * nb;
  if (nb <= 1 || items > (1 << 18) || p.n_split != 1) return nb;
  std::vector<int> w(p.n_qg);
  for (int x = 0; x < p.n_qg; ++x) w[x] = item_steps(p, qt, p.qg_desc ? p.n_qg - 1 - x : x, bc) + 2;
  std::vector<int> cand;
  for (int hb = 1; hb < nb; hb *= 2) cand.push_back(hb);
  cand.push_back(nb);
  std::vector<double> eff(cand.size());
  std::vector<long long> load(G);
  double best = 0.0;
  for (size_t k = 0; k < cand.size(); ++k) {
    const int hb = cand[k];
    std::fill(load.begin(), load.end(), 0ll);
    long long idx = 0, total = 0;
    for (int b0 = 0; b0 < nb; b0 += hb) {
      const int hbb = std::min(hb, nb - b0);
      for (int x = 0; x < p.n_qg; ++x)
        for (int h = 0; h < hbb; ++h, ++idx) {
          const long long r = idx / G, c = idx % G;
          load[(r & 1) ? G - 1 - c : c] += w[x];
          total += w[x];
        }
    }
    const long long mk = *std::max_element(load.begin(), load.end());
    eff[k] = mk > 0 ? static_cast<double>(total) / G / mk : 1.0;
    best = std::max(best, eff[k]);
  }
  int pick = -1;
  for (size_t k = 0; k < cand.size(); ++k)
    if (eff[k] >= 0.97 * best && cand[k] * kv_head <= (64ll << 20)) pick = static_cast<int>(k);
  if (pick < 0)
    for (size_t k = 0; k < cand.size(); ++k)
      if (eff[k] == best) pick = static_cast<int>(k);
  return cand[pick];
}

// Work items of the persistent forward grid: (query-tile group, split, head).
// A mask makes the query-tile groups' work unequal, so the items then go out
// group by group, heaviest groups first (with the snake order of the CTAs the
// totals even out); without one, head by head, so the query tiles of a head
// run side by side and share its K/V tiles in L2.  Each launch covers fewer
// than 2^31 items (32-bit index arithmetic in the kernel); a larger problem is
// cut into launches over ranges of heads (or of splits, if one head alone has
// that many items).  The grid has one CTA per SM (max_ctas CTAs if > 0), never
// more than the launch's items.  launch(p, grid) issues one launch.
template <class Launch>
cudaError_t launch_items(fa::FwdParams p, int qt, int bc, int d_bytes_per_row, int num_sms,
                         int max_ctas, Launch&& launch) {
  constexpr long long kMaxItems = 0x7fffffffLL;
  p.n_qg = (p.Nq + 128 * qt - 1) / (128 * qt);
  p.qg_major = (p.wl >= 0 || p.wr >= 0) ? 1 : 0;
  p.qg_desc = p.wr >= 0 ? 1 : 0;  // a right bound: later query rows see more keys
  const long long kv_head = 2ll * p.Nk * d_bytes_per_row;  // K and V of one head
  const long long per_head = static_cast<long long>(p.n_qg) * p.n_splits;
  const int heads_per = per_head > kMaxItems ? 1 : static_cast<int>(std::min<long long>(p.BH, kMaxItems / per_head));
  const int splits_per = per_head > kMaxItems ? static_cast<int>(kMaxItems / p.n_qg) : p.n_splits;
  for (int bh0 = 0; bh0 < p.BH; bh0 += heads_per) {
    for (int s0 = 0; s0 < p.n_splits; s0 += splits_per) {
      p.bh0 = bh0;
      p.n_bh = std::min(heads_per, p.BH - bh0);
      p.split0 = s0;
      p.n_split = std::min(splits_per, p.n_splits - s0);
      const long long items = static_cast<long long>(p.n_qg) * p.n_split * p.n_bh;
      p.n_items = static_cast<int>(items);
      long long g = max_ctas > 0 ? max_ctas : (num_sms > 0 ? num_sms : 1);
      if (g > items) g = items;
      p.rounds = static_cast<int>((items + g - 1) / g);
      p.hb = p.qg_major ? choose_heads_blk(p, qt, bc, static_cast<int>(g), kv_head) : p.n_bh;
#ifdef FA_HEADS_BLK
      p.hb = std::min(FA_HEADS_BLK, p.n_bh);
#endif
      p.div_qg = fa::make_fastdiv(p.n_qg);
      p.div_split = fa::make_fastdiv(p.n_split);
      p.div_blk = fa::make_fastdiv(p.n_qg * p.n_split * p.hb);
      p.div_per = fa::make_fastdiv(p.n_split * p.hb);
      const int last = p.n_bh - (p.n_bh - 1) / p.hb * p.hb;  // heads in the last block
      p.div_per_last = fa::make_fastdiv(p.n_split * last);
      const cudaError_t e = launch(p, dim3(static_cast<unsigned>(g)));
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

// fa_fwd's own split-KV workspace: m and l in fp32, O_s / l_s in bf16 (the
// merge upcasts it exactly; fa_fwd_partial's public triples stay fp32).
struct SplitLayout {
  size_t m_off, l_off, o_off, total;
};

SplitLayout split_layout(long long rows, int d, int n_splits) {
  SplitLayout L;
  const size_t ml = align256(static_cast<size_t>(n_splits) * rows * sizeof(float));
  L.m_off = 0;
  L.l_off = ml;
  L.o_off = 2 * ml;
  L.total = 2 * ml + align256(static_cast<size_t>(n_splits) * rows * d * 2);
  return L;
}

// Shared body of fa_fwd / fa_fwd_ex / fa_fwd_partial.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
             int Nk, int d, float scale, int wl, int wr, int n_splits, void* stream,
             const fa_opts* opts, float* m_part, float* l_part, float* o_part,
             void* split_ws = nullptr, size_t split_ws_bytes = 0) {
  const bool partial = (m_part != nullptr);
  int rc = check_sizes(B, H, Nq, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (!q || !k || !v) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return FA_ERR_INVALID_ARG;
  if (partial) {
    if (!l_part || !o_part || !aligned(m_part, 4) || !aligned(l_part, 4) || !aligned(o_part, 16))
      return FA_ERR_INVALID_ARG;
  } else {
    if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  }
  if (n_splits < 1 || n_splits > 65535) return FA_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1 || wl > kMaxSeq || wr > kMaxSeq) return FA_ERR_INVALID_ARG;
  int bc = fa::kDefaultBc, qt_opt = 0, skip = -1, max_ctas = 0;
  unsigned long long timeout = kDefaultTimeoutNs;
  if (opts) {
    if (opts->bc != 0 && opts->bc != 64 && opts->bc != 128) return FA_ERR_INVALID_ARG;
    if (opts->q_tiles_per_cta < 0 || opts->q_tiles_per_cta > 2) return FA_ERR_INVALID_ARG;
    if (opts->test_skip_kv_load < 0 || opts->max_ctas < 0) return FA_ERR_INVALID_ARG;
    if (opts->bc) bc = opts->bc;
    qt_opt = opts->q_tiles_per_cta;
    if (opts->timeout_ns) timeout = opts->timeout_ns;
    skip = opts->test_skip_kv_load - 1;
    max_ctas = opts->max_ctas;
  }
  DevState* dev = nullptr;
  if ((rc = device_state(&dev)) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const int BH = B * H;
  const int kv_tiles = (Nk + bc - 1) / bc;
  const int qt = qt_opt ? qt_opt : (Nq > 128 ? 2 : 1);
  int splits = n_splits;
  if (!partial && splits > kv_tiles) splits = kv_tiles;

  fa::FwdParams p{};
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = BH;
  p.n_splits = partial ? splits : (splits > 1 ? splits : 1);
  p.partial = (partial || splits > 1) ? 1 : 0;
  p.kv_tiles = kv_tiles;
  p.tiles_per_split = (kv_tiles + splits - 1) / splits;
  p.wl = wl;
  p.wr = wr;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = timeout;
  p.test_skip_load = skip;
  p.status = dev->status;
  p.o = o;
  p.lse = lse;

  CUtensorMap maps[4];
  if ((rc = make_map(&maps[0], q, d, Nq, BH, 128)) != FA_OK) return rc;
  if ((rc = make_map(&maps[1], k, d, Nk, BH, bc)) != FA_OK) return rc;
  if ((rc = make_map(&maps[2], v, d, Nk, BH, bc)) != FA_OK) return rc;
  if (!partial && splits == 1) {
    if ((rc = make_map(&maps[3], o, d, Nq, BH, 128)) != FA_OK) return rc;
  } else {
    maps[3] = maps[0];  // unused by the partial epilogue
  }
  const long long rows = static_cast<long long>(BH) * Nq;
  auto run = [&](const fa::FwdParams& pp) {
    return launch_items(pp, qt, bc, d * 2, dev->num_sms, max_ctas, [&](const fa::FwdParams& pl, dim3 grid) {
      return launch_fwd(d, bc, qt, maps, pl, grid, s);
    });
  };

  if (partial) {
    p.m_part = m_part;
    p.l_part = l_part;
    p.o_part = o_part;
    cudaError_t e = run(p);
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }
  if (splits == 1) {
    cudaError_t e = run(p);
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }

  // split-KV: workspace (stream-ordered, or the caller's), partial kernel,
  // merge, release
  const SplitLayout L = split_layout(rows, d, splits);
  void* ws = split_ws;
  cudaError_t e = cudaSuccess;
  if (ws) {
    if (split_ws_bytes < L.total) return FA_ERR_SCRATCH_TOO_SMALL;
  } else if ((e = cudaMallocAsync(&ws, L.total, s)) != cudaSuccess) {
    t_last_cuda = e;
    return FA_ERR_NO_MEMORY;
  }
  char* base = static_cast<char*>(ws);
  p.m_part = reinterpret_cast<float*>(base + L.m_off);
  p.l_part = reinterpret_cast<float*>(base + L.l_off);
  p.o_part = base + L.o_off;
  p.part_bf16 = 1;
  e = run(p);
  if (e == cudaSuccess) {
    fa::MergeParams mp{};
    mp.m_part = p.m_part;
    mp.l_part = p.l_part;
    mp.o_part = p.o_part;
    mp.o_part_bf16 = 1;
    mp.o = o;
    mp.lse = lse;
    mp.rows = rows;
    mp.n_splits = splits;
    e = fa::launch_merge(d, mp, s);
  }
  const cudaError_t ef = split_ws ? cudaSuccess : cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (ef != cudaSuccess) return cuda_fail(ef);
  return FA_OK;
}

// fa_fwd_host: per-device device buffer and streams, held across calls.
constexpr int kMaxHostChunks = 64;
constexpr int kHostRunStreams = 2;  // kernel streams of the host pipeline, used in turn
struct HostPipe {
  std::mutex mu;
  bool init = false;
  char* buf = nullptr;
  size_t cap = 0;
  cudaStream_t s_in = nullptr, s_run[kHostRunStreams] = {}, s_out = nullptr;
  cudaEvent_t in_done[kMaxHostChunks], run_done[kMaxHostChunks];
};

// Head groups of the host pipeline: n_chunks > 0 gives that many groups of
// equal size (clamped to [1, min(BH, kMaxHostChunks)]); otherwise groups of
// a quarter of the heads, then halving toward the end (64 heads: 16, 16, 16,
// 8, 4, 2, 2), so the copies in run in few large transfers while the last
// group -- whose kernel and copy out nothing overlaps -- is small.  Returns
// the number of groups; sizes[g] heads in group g.
int host_groups(int BH, int n_chunks, int* sizes) {
  int n = 0;
  if (n_chunks > 0) {
    int chunks = std::min(std::min(n_chunks, BH), kMaxHostChunks);
    const int per = (BH + chunks - 1) / chunks;
    for (int h0 = 0; h0 < BH; h0 += per) sizes[n++] = std::min(per, BH - h0);
    return n;
  }
  const int big = std::max(1, (BH + 3) / 4);
  int rest = BH;
  while (rest > 2 * big) sizes[n++] = big, rest -= big;
  while (rest > 2) {
    const int g = (rest + 1) / 2;
    sizes[n++] = g;
    rest -= g;
  }
  if (rest > 0) sizes[n++] = rest;
  return n;
}
HostPipe g_pipe[kMaxDevices];

int host_pipe_init(HostPipe& hp) {
  if (hp.init) return FA_OK;
  cudaError_t e = cudaSuccess;
  for (cudaStream_t* st : {&hp.s_in, &hp.s_out})
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
  for (cudaStream_t& st : hp.s_run)
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  for (int c = 0; e == cudaSuccess && c < kMaxHostChunks; ++c) {
    e = cudaEventCreateWithFlags(&hp.in_done[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.run_done[c], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  hp.init = true;
  return FA_OK;
}

}  // namespace

namespace fa {
// fa_fwd with n_splits > 1 and its workspace in the caller's device memory
// (ws_bytes of it, FA_ERR_SCRATCH_TOO_SMALL if the split layout needs more).
int fwd_split_into(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Nq, int Nk, int d, float scale, int causal, int n_splits, void* stream,
                   void* ws, size_t ws_bytes) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_splits, stream,
                  nullptr, nullptr, nullptr, nullptr, ws, ws_bytes);
}
}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
           int Nk, int d, float scale, int causal, int n_splits, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_splits, stream,
                  nullptr, nullptr, nullptr, nullptr);
}

// fa_fwd_host / fa_fwd_local_host / fa_fwd_fp8_host: the forward with mask
// (wl, wr) on host buffers; fp8 = the three descales of the E4M3 forward (one
// byte per Q, K, V element; O stays bf16), or nullptr for bf16.
static int fwd_host_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int Nq, int Nk, int d, float scale, int wl, int wr, int n_chunks,
                         const float* fp8) {
  int rc = check_sizes(B, H, Nq, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1 || wl > kMaxSeq || wr > kMaxSeq) return FA_ERR_INVALID_ARG;
  if (fp8) {
    if (d != 128) return FA_ERR_UNSUPPORTED;
    for (int i = 0; i < 3; ++i)
      if (!std::isfinite(fp8[i]) || !(fp8[i] > 0.f)) return FA_ERR_INVALID_ARG;
  }
  DevState* dev = nullptr;
  if ((rc = device_state(&dev)) != FA_OK) return rc;
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return cuda_fail(e);
  HostPipe& hp = g_pipe[dev_id];
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((rc = host_pipe_init(hp)) != FA_OK) return rc;

  const int BH = B * H;
  const size_t in_es = fp8 ? 1 : 2;  // bytes per Q, K, V element
  const size_t q_head = static_cast<size_t>(Nq) * d * in_es, kv_head = static_cast<size_t>(Nk) * d * in_es;
  const size_t o_head = static_cast<size_t>(Nq) * d * 2, lse_head = static_cast<size_t>(Nq) * 4;
  const size_t off_k = align256(BH * q_head), off_v = off_k + align256(BH * kv_head);
  const size_t off_o = off_v + align256(BH * kv_head), off_l = off_o + align256(BH * o_head);
  const size_t need = off_l + align256(BH * lse_head);
  if (need > hp.cap) {
    if (hp.buf && (e = cudaFree(hp.buf)) != cudaSuccess) return cuda_fail(e);
    hp.buf = nullptr;
    hp.cap = 0;
    if ((e = cudaMalloc(&hp.buf, need)) != cudaSuccess) {
      t_last_cuda = e;
      return FA_ERR_NO_MEMORY;
    }
    hp.cap = need;
  }
  char* dq = hp.buf;
  char* dk = hp.buf + off_k;
  char* dv = hp.buf + off_v;
  char* dout = hp.buf + off_o;
  float* dl = reinterpret_cast<float*>(hp.buf + off_l);
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  char* ho = static_cast<char*>(o);

  int sizes[kMaxHostChunks];
  const int groups = host_groups(BH, n_chunks, sizes);
  // Group c: its heads' copies in on s_in, the kernel on s_run[c %
  // kHostRunStreams] after them (kernel streams in turn, so a small group's
  // kernel need not wait for the previous group's), copies out on s_out after
  // the kernel.  (A second
  // copy-in stream gained nothing: one stream already fills the
  // host-to-device link, about 205 GB/s on GB300.)
  for (int c = 0, h0 = 0; c < groups && rc == FA_OK && e == cudaSuccess; h0 += sizes[c++]) {
    const int nh = sizes[c];
    cudaStream_t si = hp.s_in, sr = hp.s_run[c % kHostRunStreams];
    e = cudaMemcpyAsync(dq + h0 * q_head, hq + h0 * q_head, nh * q_head, cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dk + h0 * kv_head, hk + h0 * kv_head, nh * kv_head, cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dv + h0 * kv_head, hv + h0 * kv_head, nh * kv_head, cudaMemcpyHostToDevice, si);
    if (e == cudaSuccess) e = cudaEventRecord(hp.in_done[c], si);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sr, hp.in_done[c], 0);
    if (e != cudaSuccess) break;
    if (fp8)
      rc = fa_fwd_fp8(dq + h0 * q_head, dk + h0 * kv_head, dv + h0 * kv_head, dout + h0 * o_head,
                      dl + static_cast<size_t>(h0) * Nq, 1, nh, Nq, Nk, d, scale, fp8[0], fp8[1], fp8[2],
                      wr == 0 ? 1 : 0, sr);
    else
      rc = fwd_impl(dq + h0 * q_head, dk + h0 * kv_head, dv + h0 * kv_head, dout + h0 * o_head,
                    dl + static_cast<size_t>(h0) * Nq, 1, nh, Nq, Nk, d, scale, wl, wr, 1, sr, nullptr,
                    nullptr, nullptr, nullptr);
    if (rc != FA_OK) break;
    e = cudaEventRecord(hp.run_done[c], sr);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.s_out, hp.run_done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ho + h0 * o_head, dout + h0 * o_head, nh * o_head, cudaMemcpyDeviceToHost,
                          hp.s_out);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(lse + static_cast<size_t>(h0) * Nq, dl + static_cast<size_t>(h0) * Nq,
                          nh * lse_head, cudaMemcpyDeviceToHost, hp.s_out);
  }
  // drain every stream whatever happened above
  cudaError_t es = cudaStreamSynchronize(hp.s_in);
  cudaError_t er = cudaSuccess;
  for (cudaStream_t st : hp.s_run) {
    const cudaError_t x = cudaStreamSynchronize(st);
    if (er == cudaSuccess) er = x;
  }
  cudaError_t eo = cudaStreamSynchronize(hp.s_out);
  if (rc != FA_OK) return rc;
  if (e != cudaSuccess) return cuda_fail(e);
  if (es != cudaSuccess) return cuda_fail(es);
  if (er != cudaSuccess) return cuda_fail(er);
  if (eo != cudaSuccess) return cuda_fail(eo);
  return fa_get_device_status(hp.s_out);
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, float scale, int causal, int n_chunks) {
  return fwd_host_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_chunks, nullptr);
}

int fa_fwd_local_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, float scale, int window_left, int window_right,
                      int n_chunks) {
  return fwd_host_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, window_left, window_right, n_chunks,
                       nullptr);
}

int fa_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                    float v_descale, int causal, int n_chunks) {
  const float ds[3] = {q_descale, k_descale, v_descale};
  return fwd_host_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_chunks, ds);
}

int fa_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Nq, int Nk, int d, float scale, int window_left, int window_right, int n_splits,
                 void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, window_left, window_right, n_splits,
                  stream, nullptr, nullptr, nullptr, nullptr);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, int n_splits, void* stream,
              const fa_opts* opts) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_splits, stream,
                  opts, nullptr, nullptr, nullptr);
}

int fa_fwd_partial(const void* q, const void* k, const void* v, float* m_part, float* l_part,
                   float* o_part, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   int n_splits, void* stream) {
  if (!m_part) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, nullptr, nullptr, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1, n_splits,
                  stream, nullptr, m_part, l_part, o_part);
}

int fa_merge_splits(const float* m_part, const float* l_part, const float* o_part, void* o,
                    float* lse, int B, int H, int Nq, int d, int n_splits, void* stream) {
  if (B < 1 || H < 1 || Nq < 1 || Nq > kMaxSeq) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (n_splits < 1 || n_splits > 65535) return FA_ERR_INVALID_ARG;
  if (!m_part || !l_part || !o_part || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(o, 16) || !aligned(m_part, 4) || !aligned(l_part, 4) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != FA_OK) return rc;
  fa::MergeParams mp{};
  mp.m_part = m_part;
  mp.l_part = l_part;
  mp.o_part = o_part;
  mp.o = o;
  mp.lse = lse;
  mp.rows = static_cast<long long>(B) * H * Nq;
  mp.n_splits = n_splits;
  cudaError_t e = fa::launch_merge(d, mp, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
               float v_descale, int causal, void* stream) {
  int rc = check_sizes(B, H, Nq, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  for (float x : {q_descale, k_descale, v_descale})
    if (!std::isfinite(x) || !(x > 0.f)) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  if ((rc = device_state(&dev)) != FA_OK) return rc;
  const int BH = B * H;
  const int qt = Nq > 128 ? 2 : 1;
  fa::FwdParams p{};
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = BH;
  p.n_splits = 1;
  p.partial = 0;
  p.kv_tiles = (Nk + 127) / 128;
  p.tiles_per_split = p.kv_tiles;
  p.wl = -1;
  p.wr = causal ? 0 : -1;
  const double s_qk = static_cast<double>(scale) * q_descale * k_descale;
  p.scale = static_cast<float>(s_qk);
  p.scale_log2 = static_cast<float>(s_qk * 1.4426950408889634);
  p.o_scale = v_descale / 256.f;  // final_scale
  p.timeout_ns = kDefaultTimeoutNs;
  p.test_skip_load = -1;
  p.status = dev->status;
  p.o = o;
  p.lse = lse;
  CUtensorMap maps[4];
  if ((rc = make_map(&maps[0], q, d, Nq, BH, 128, true)) != FA_OK) return rc;
  if ((rc = make_map(&maps[1], k, d, Nk, BH, 128, true)) != FA_OK) return rc;
  if ((rc = make_map(&maps[2], v, d, Nk, BH, 128, true)) != FA_OK) return rc;
  if ((rc = make_map(&maps[3], o, d, Nq, BH, 128)) != FA_OK) return rc;
  cudaError_t e = launch_items(p, qt, 128, d, dev->num_sms, 0, [&](const fa::FwdParams& pl, dim3 grid) {
    return fa::launch_fwd_fp8_d128(qt, maps, pl, grid, static_cast<cudaStream_t>(stream));
  });
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

// Shared body of fa_bwd / fa_bwd_local.
static int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                    int d, float scale, int wl, int wr, void* stream) {
  int rc = check_sizes(B, H, Nq, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (wl < -1 || wr < -1 || wl > kMaxSeq || wr > kMaxSeq) return FA_ERR_INVALID_ARG;
  const void* in[6] = {q, k, v, o, dout, lse};
  void* out[3] = {dq, dk, dv};
  for (const void* ptr : in)
    if (!ptr) return FA_ERR_INVALID_ARG;
  for (void* ptr : out)
    if (!ptr || !aligned(ptr, 16)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  if ((rc = device_state(&dev)) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const int nq_pad = (Nq + 127) / 128 * 128;

  CUtensorMap maps[7];  // q, k, v, dout, dq, dk, dv
  const void* bases[7] = {q, k, v, dout, dq, dk, dv};
  const int rows[7] = {Nq, Nk, Nk, Nq, Nq, Nk, Nk};
  for (int i = 0; i < 7; ++i)
    if ((rc = make_map(&maps[i], bases[i], d, rows[i], BH, 128)) != FA_OK) return rc;

  const size_t vec = align256(static_cast<size_t>(BH) * nq_pad * sizeof(float));
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, 2 * vec, s);
  if (e != cudaSuccess) {
    t_last_cuda = e;
    return FA_ERR_NO_MEMORY;
  }
  fa::BwdPreParams pre{};
  pre.o = o;
  pre.dout = dout;
  pre.lse = lse;
  pre.nlse2 = static_cast<float*>(ws);
  pre.nd = reinterpret_cast<float*>(static_cast<char*>(ws) + vec);
  pre.Nq = Nq;
  pre.nq_pad = nq_pad;
  pre.BH = BH;
  fa::BwdParams p{};
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = BH;
  p.nq_pad = nq_pad;
  p.wl = wl;
  p.wr = wr;
  p.causal = (wl < 0 && wr >= 0) ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.nlse2 = pre.nlse2;
  p.nd = pre.nd;
  p.timeout_ns = kDefaultTimeoutNs;
  p.status = dev->status;
  e = d == 64 ? fa::launch_bwd_d64(maps, p, pre, s) : fa::launch_bwd_d128(maps, p, pre, s);
  cudaError_t e2 = cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (e2 != cudaSuccess) return cuda_fail(e2);
  return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
           float scale, int causal, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1,
                  stream);
}

int fa_bwd_local(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                 int d, float scale, int window_left, int window_right, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, window_left,
                  window_right, stream);
}

// fa_bwd_host / fa_bwd_local_host: the backward on host buffers, through the
// head-group pipeline of fa_fwd_host (six copies in, the backward, three out).
static int bwd_host_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                         int d, float scale, int wl, int wr, int n_chunks) {
  int rc = check_sizes(B, H, Nq, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1 || wl > kMaxSeq || wr > kMaxSeq) return FA_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  if ((rc = device_state(&dev)) != FA_OK) return rc;
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return cuda_fail(e);
  HostPipe& hp = g_pipe[dev_id];
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((rc = host_pipe_init(hp)) != FA_OK) return rc;

  const int BH = B * H;
  // per head: bytes of each array, in the order in[] / out[] list them
  const size_t q_head = static_cast<size_t>(Nq) * d * 2, kv_head = static_cast<size_t>(Nk) * d * 2;
  const size_t lse_head = static_cast<size_t>(Nq) * 4;
  const size_t in_head[6] = {q_head, kv_head, kv_head, q_head, q_head, lse_head};  // q k v o dout lse
  const size_t out_head[3] = {q_head, kv_head, kv_head};                            // dq dk dv
  size_t off_in[6], off_out[3], need = 0;
  for (int a = 0; a < 6; ++a) off_in[a] = need, need += align256(BH * in_head[a]);
  for (int a = 0; a < 3; ++a) off_out[a] = need, need += align256(BH * out_head[a]);
  if (need > hp.cap) {
    if (hp.buf && (e = cudaFree(hp.buf)) != cudaSuccess) return cuda_fail(e);
    hp.buf = nullptr;
    hp.cap = 0;
    if ((e = cudaMalloc(&hp.buf, need)) != cudaSuccess) {
      t_last_cuda = e;
      return FA_ERR_NO_MEMORY;
    }
    hp.cap = need;
  }
  const char* h_in[6] = {static_cast<const char*>(q), static_cast<const char*>(k),
                         static_cast<const char*>(v), static_cast<const char*>(o),
                         static_cast<const char*>(dout), reinterpret_cast<const char*>(lse)};
  char* h_out[3] = {static_cast<char*>(dq), static_cast<char*>(dk), static_cast<char*>(dv)};

  int sizes[kMaxHostChunks];
  const int groups = host_groups(BH, n_chunks, sizes);
  for (int c = 0, h0 = 0; c < groups && rc == FA_OK && e == cudaSuccess; h0 += sizes[c++]) {
    const int nh = sizes[c];
    cudaStream_t sr = hp.s_run[c % kHostRunStreams];
    char* d_in[6];
    char* d_out[3];
    for (int a = 0; a < 6; ++a) d_in[a] = hp.buf + off_in[a] + h0 * in_head[a];
    for (int a = 0; a < 3; ++a) d_out[a] = hp.buf + off_out[a] + h0 * out_head[a];
    for (int a = 0; a < 6 && e == cudaSuccess; ++a)
      e = cudaMemcpyAsync(d_in[a], h_in[a] + h0 * in_head[a], nh * in_head[a], cudaMemcpyHostToDevice,
                          hp.s_in);
    if (e == cudaSuccess) e = cudaEventRecord(hp.in_done[c], hp.s_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sr, hp.in_done[c], 0);
    if (e != cudaSuccess) break;
    rc = bwd_impl(d_in[0], d_in[1], d_in[2], d_in[3], reinterpret_cast<const float*>(d_in[5]), d_in[4],
                  d_out[0], d_out[1], d_out[2], 1, nh, Nq, Nk, d, scale, wl, wr, sr);
    if (rc != FA_OK) break;
    e = cudaEventRecord(hp.run_done[c], sr);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.s_out, hp.run_done[c], 0);
    for (int a = 0; a < 3 && e == cudaSuccess; ++a)
      e = cudaMemcpyAsync(h_out[a] + h0 * out_head[a], d_out[a], nh * out_head[a], cudaMemcpyDeviceToHost,
                          hp.s_out);
  }
  // drain every stream whatever happened above
  cudaError_t es = cudaStreamSynchronize(hp.s_in);
  cudaError_t er = cudaSuccess;
  for (cudaStream_t st : hp.s_run) {
    const cudaError_t x = cudaStreamSynchronize(st);
    if (er == cudaSuccess) er = x;
  }
  cudaError_t eo = cudaStreamSynchronize(hp.s_out);
  if (rc != FA_OK) return rc;
  if (e != cudaSuccess) return cuda_fail(e);
  if (es != cudaSuccess) return cuda_fail(es);
  if (er != cudaSuccess) return cuda_fail(er);
  if (eo != cudaSuccess) return cuda_fail(eo);
  return fa_get_device_status(hp.s_out);
}

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                float scale, int causal, int n_chunks) {
  return bwd_host_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, -1, causal ? 0 : -1,
                       n_chunks);
}

int fa_bwd_local_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                      int d, float scale, int window_left, int window_right, int n_chunks) {
  return bwd_host_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, window_left,
                       window_right, n_chunks);
}

int fa_softmax_rows(const void* x, void* y, float* lse, long long rows, int cols, int dtype,
                    void* stream) {
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (rows < 0 || cols < 1 || cols > kMaxSeq) return FA_ERR_INVALID_ARG;
  const size_t elt = dtype == FA_DTYPE_F32 ? 4 : 2;
  if (rows > 0 && (!x || !y || !aligned(x, elt) || !aligned(y, elt) || (lse && !aligned(lse, 4))))
    return FA_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != FA_OK) return rc;
  if (rows == 0) return FA_OK;
  fa::SoftmaxParams p{};
  p.x = x;
  p.y = y;
  p.lse = lse;
  p.rows = rows;
  p.cols = cols;
  p.status = dev->status;
  p.timeout_ns = kDefaultTimeoutNs;
  // 16-byte vectors when every row starts on a 16-byte boundary
  const bool vec = aligned(x, 16) && aligned(y, 16) && (static_cast<size_t>(cols) * elt) % 16 == 0;
  cudaError_t e = fa::launch_softmax_rows(p, dtype == FA_DTYPE_BF16, vec, dev->num_sms,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

size_t fa_split_workspace_bytes(int B, int H, int Nq, int d, int n_splits) {
  if (B < 1 || H < 1 || Nq < 1 || n_splits <= 1 || (d != 64 && d != 128)) return 0;
  return split_layout(static_cast<long long>(B) * H * Nq, d, n_splits).total;
}

int fa_get_device_status(void* stream) {
  DevState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host[2] = {0, 0};
  const int zero[2] = {0, 0};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, dev->status, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (host[0] == fa::kDevCheck) {
    std::snprintf(t_check_msg, sizeof(t_check_msg),
                  "debug build: a device-side bounds check failed (kernel source line %d); the "
                  "access was skipped",
                  host[1]);
    return FA_ERR_DEVICE_CHECK;
  }
  if (host[0] == fa::kDevLayout) return FA_ERR_UNSUPPORTED;
  return host[0] == fa::kDevTimeout ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported (head dim must be 64 or 128; device must be sm_103)";
    case FA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out; the affected CTAs stopped without writing";
    case FA_ERR_DEVICE_CHECK: return t_check_msg;
    case FA_ERR_NO_MEMORY: return "could not allocate the split-KV workspace";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "split-KV workspace larger than the fixed no-alloc scratch (FA_NOALLOC_SCRATCH_BYTES)";
    case FA_ERR_CUDA:
      std::snprintf(t_msg, sizeof(t_msg), "CUDA error %d: %s", static_cast<int>(t_last_cuda),
                    cudaGetErrorString(t_last_cuda));
      return t_msg;
    default: return "unknown error code";
  }
}

int fa_version(void) { return kVersion; }

}  // extern "C"
