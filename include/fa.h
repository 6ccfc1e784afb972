/*
 * fa.h -- C ABI of the single-pass online-softmax attention forward for
 * NVIDIA GB300 (sm_103a).  Library: libfa.so.
 *
 * Operation (all entry points): for each batch b, head h and query row i,
 *
 *   S_ij  = scale * <q[b,h,i,:], k[b,h,j,:]>      (-inf where masked)
 *   O_i   = sum_j softmax_j(S_i) v[b,h,j,:]
 *   LSE_i = ln sum_j exp(S_ij)                     (natural log)
 *
 * computed in one pass over K/V tiles with the online-softmax recurrence
 * (running max m, running sum l, rescaled accumulator O, one division by l at
 * the end): "Online Softmax 算法详解" (inference.lei6393.com) sections 2.3, 3.2,
 * 4.7 and 8.1; "在线Softmax算法解析：FlashAttention核心技术" (intelliparadigm.com)
 * section 3.2; "01 -- La recurrencia del online softmax" (lynx-cortex.pages.dev),
 * section "La recurrencia".
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, in device memory (cudaMalloc / caching
 *     allocator memory of the current device).  The caller owns every buffer;
 *     the library keeps no pointer after the call returns.
 *   - q, k, v, o: bf16 [B][H][N][d] with N = Nq for q/o and Nk for k/v;
 *     base addresses 16-byte aligned.  lse: fp32 [B][H][Nq].
 *   - d in {64, 128}; 1 <= Nq, Nk <= 2^30; B*H <= 65535; scale finite and > 0
 *     (the usual value is 1/sqrt(d)).
 *   - causal != 0: key j is visible to query i iff j <= i + (Nk - Nq)
 *     (bottom-right alignment; equal to j <= i when Nq == Nk).  A query row
 *     that sees no key gets O = 0 and LSE = -inf ("Online Softmax 算法详解"
 *     sections 7.2-7.3).
 *   - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on it; buffers must stay valid until the work
 *     on `stream` completes.  The calling thread's current device must be the
 *     device that owns the buffers and the stream.
 *   - Return value: FA_OK (0), or a negative FA_ERR_* code.  Argument errors
 *     are detected before anything is launched; on error nothing is written.
 *     The library never aborts the process and never traps on the device.
 *   - Device-side timeouts: every wait inside the kernels is bounded.  A wait
 *     that runs out stops its CTA cleanly (outputs of that CTA are left
 *     unwritten) and records FA_ERR_DEVICE_TIMEOUT, which
 *     fa_get_device_status() reports.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_INVALID_ARG (-1)    /* null/misaligned pointer, bad size, bad scale */
#define FA_ERR_UNSUPPORTED (-2)    /* d not in {64,128}, device is not sm_103, or (from
                                      fa_get_device_status) a shared memory base the
                                      backward's layout cannot use */
#define FA_ERR_CUDA (-3)           /* a CUDA call failed; fa_strerror() has details */
#define FA_ERR_DEVICE_TIMEOUT (-4) /* a kernel wait ran out (fa_get_device_status) */
#define FA_ERR_NO_MEMORY (-5)      /* the split-KV workspace could not be allocated */
#define FA_ERR_SCRATCH_TOO_SMALL (-6) /* fa_fwd_split_noalloc: workspace over the fixed limit */
#define FA_ERR_DEVICE_CHECK (-7)   /* debug build (libfa_debug.so) only: a device-side bounds
                                      check failed (fa_get_device_status; fa_strerror gives
                                      the kernel source line) */

/*
 * Attention forward, O and LSE.
 *
 * n_splits == 1: one kernel, each CTA walks the whole key axis and writes O
 *   (bf16) and LSE (fp32) directly.
 * n_splits  > 1: split-KV.  The key axis is cut into n_splits contiguous
 *   ranges of K/V tiles (clamped to the number of 128-key tiles); each range
 *   yields a partial (m, l, O) triple per row, combined by the two-block merge
 *   rule (see fa_merge_splits).  The workspace for the partials (m and l in
 *   fp32, O_s / l_s rounded to bf16: half the bytes of fa_fwd_partial's fp32
 *   triples through HBM, written and read back) is taken with
 *   cudaMallocAsync on `stream` and released with cudaFreeAsync on the same
 *   stream (FA_ERR_NO_MEMORY if that fails).  The bf16 partials add at most
 *   2^-8 max_s |O_s| to each element of O before its own bf16 rounding.
 *
 * q, k, v : in,  bf16 [B][H][Nq|Nk][d]
 * o       : out, bf16 [B][H][Nq][d]
 * lse     : out, fp32 [B][H][Nq], natural-log units of the scaled logits:
 *           LSE_i = scale*m_i + ln l_i ("Online Softmax 算法详解" section 8.2).
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
           int Nk, int d, float scale, int causal, int n_splits, void* stream);

/*
 * fa_fwd on HOST buffers, the copies included: Q, K, V go to the device, the
 * forward runs, O and LSE come back; returns once o and lse hold the result.
 * The (b, h) heads are cut into groups of consecutive heads that pass through
 * internal streams (host-to-device copies; kernels, on two streams used in
 * turn; device-to-host copies), so one group's copies overlap other groups'
 * kernels.  n_chunks > 0: that many groups of equal size (clamped to
 * min(B*H, 64)).  n_chunks <= 0: groups of a quarter of the heads, then
 * halving toward the end (64 heads: 16, 16, 16, 8, 4, 2, 2) -- few large
 * copies in, and a small last group, whose kernel and copy out nothing
 * overlaps.  Every grouping gives the same bits as fa_fwd.
 *
 * q, k, v : in,  host bf16 [B][H][Nq|Nk][d]
 * o       : out, host bf16 [B][H][Nq][d]
 * lse     : out, host fp32 [B][H][Nq]
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to run asynchronously and overlap; pageable buffers give the same
 * results, staged by the driver.  Device memory: one buffer per device of the
 * problem's size (Q, K, V, O, LSE), kept by the library for later calls and
 * grown when a larger call comes (FA_ERR_NO_MEMORY if that fails).  Calls on
 * the same device are serialised (they share that buffer and the streams).
 * Errors: as fa_fwd; FA_ERR_DEVICE_TIMEOUT if a device-side wait ran out.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, float scale, int causal, int n_chunks);

/*
 * Attention forward with a local (sliding-window) mask, "causal, local" masks
 * of "Online Softmax 算法详解" section 3.2 (which names the local mask without
 * defining it).  With off = Nk - Nq, key j is visible to query i iff
 *   i + off - window_left <= j <= i + off + window_right,
 * and a bound of -1 leaves that side open: (-1, 0) is fa_fwd's causal mask and
 * (-1, -1) the unmasked forward.  K/V tiles wholly outside a query tile's
 * window are skipped.  Rows that see no key get O = 0 and LSE = -inf.
 * Arguments otherwise as fa_fwd (n_splits > 1 = split-KV with merge);
 * window_left, window_right in [-1, 2^30].
 */
int fa_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Nq, int Nk, int d, float scale, int window_left, int window_right, int n_splits,
                 void* stream);

/*
 * fa_fwd_local on HOST buffers: the mask of fa_fwd_local (window_left,
 * window_right in [-1, 2^30]), the copies and head groups of fa_fwd_host, whose
 * buffer, stream, blocking and error rules apply unchanged.
 */
int fa_fwd_local_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, float scale, int window_left, int window_right,
                      int n_chunks);

/*
 * Attention backward from the saved LSE ("Online Softmax 算法详解" section 8.3:
 * recompute S = Q K^T, restore P = exp(scale S - LSE) without a second online
 * softmax, then form the gradients).  With D_i = <dO_i, O_i>:
 *   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (<dO_i, V_j> - D_i),
 *   dK_j = scale sum_i dS_ij Q_i,   dQ_i = scale sum_j dS_ij K_j.
 * A row with LSE = -inf (no visible key) contributes nothing (section 7.3).
 *
 * q, k, v, o : in, bf16, as fa_fwd (o = the forward's output)
 * lse        : in, fp32 [B][H][Nq], the forward's LSE
 * dout       : in, bf16 [B][H][Nq][d], gradient of the loss with respect to O
 * dq, dk, dv : out, bf16, shapes of q, k, v; 16-byte aligned
 * causal     : the mask of the forward call (bottom-right aligned)
 * Two kernels after a small row pass: one per 128-key tile (dK, dV) and one per
 * 128-query tile (dQ); S and dP are recomputed in both, and no result is
 * accumulated atomically, so repeated calls give identical bits.  A fp32
 * workspace of 2 * B*H*ceil(Nq/128)*128 floats is taken with cudaMallocAsync
 * on `stream` and released on it (FA_ERR_NO_MEMORY if that fails).
 * Arguments otherwise as fa_fwd.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
           float scale, int causal, void* stream);

/* fa_bwd for a forward run with fa_fwd_local's window (window_left, window_right). */
int fa_bwd_local(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                 int d, float scale, int window_left, int window_right, void* stream);

/*
 * fa_bwd / fa_bwd_local on HOST buffers: q, k, v, o, lse, dout in and dq, dk,
 * dv out are host arrays (layouts as fa_bwd), copied through the head-group
 * pipeline of fa_fwd_host, whose buffer, stream, blocking and error rules apply
 * unchanged.  fa_bwd_local_host takes the window of fa_fwd_local.
 */
int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                float scale, int causal, int n_chunks);
int fa_bwd_local_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                      int d, float scale, int window_left, int window_right, int n_chunks);

/*
 * FP8 (E4M3) attention forward with Max_offset = 8 ("Online Softmax 算法详解"
 * section 6).  q, k, v hold E4M3 bytes (bf16 layout, one byte per element);
 * their real values are q * q_descale, k * k_descale, v * v_descale.  The
 * online recurrence runs as in fa_fwd on S = scale q_descale k_descale Q K^T,
 * except that P' = 2^((S - m) log2(e) + 8) in [0, 256] is cast to E4M3 (round
 * to nearest even, saturating) for the P.V product; the row sum accumulates the
 * fp32 P' and is scaled by 2^-8 at the end (sum_scale), O by
 * final_scale = v_descale 2^-8.
 * o   : out, bf16 [B][H][Nq][d];  lse : out, fp32 [B][H][Nq] (natural log)
 * d must be 128 (FA_ERR_UNSUPPORTED otherwise); descales finite and > 0;
 * causal as in fa_fwd; no split-KV.  Arguments otherwise as fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
               float v_descale, int causal, void* stream);

/*
 * fa_fwd_fp8 on HOST buffers: E4M3 Q, K, V (one byte per element) in, bf16 O
 * and fp32 LSE out, with the copies and head groups of fa_fwd_host, whose
 * buffer, stream, blocking and error rules apply unchanged.  Arguments as
 * fa_fwd_fp8 (d = 128; descales finite and > 0, checked before any copy).
 */
int fa_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                    float v_descale, int causal, int n_chunks);

/* Options for fa_fwd_ex.  Zero-initialise, then set what you need. */
typedef struct fa_opts {
  int bc;                     /* K/V tile rows: 0 = default (128), or 64 or 128 */
  int q_tiles_per_cta;        /* 0 = automatic (2 when Nq > 128), or 1 or 2 */
  unsigned long long timeout_ns; /* bound of each device-side wait; 0 = 4 s */
  int test_skip_kv_load;      /* test hook: 0 = off; n > 0 makes the producer
                                 of every CTA skip its n-th K/V tile load, so
                                 the consumer's wait runs out and the call
                                 reports FA_ERR_DEVICE_TIMEOUT */
  int max_ctas;               /* 0 = one CTA per SM; n > 0: n CTAs (at most
                                 one per work item; beyond one per SM they run
                                 in waves).  Same results for every n */
} fa_opts;

/* fa_fwd with options; opts may be NULL (same as fa_fwd). */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, int n_splits, void* stream,
              const fa_opts* opts);

/*
 * Split-KV forward without the merge: writes the n_splits partial triples
 * ("the partial (m^(i), l^(i), O^(i))" of the two-block merge rule, airsota.com
 * online-softmax card, section 三).  Split s covers K/V tiles
 * [s*T', min(T, (s+1)*T')) with T = ceil(Nk/128) and T' = ceil(T/n_splits);
 * a split with no visible key yields m = -inf, l = 0, O = 0.
 *
 * m_part : out, fp32 [n_splits][B][H][Nq]   m_s = scale * (raw max), natural-log units
 * l_part : out, fp32 [n_splits][B][H][Nq]   l_s = sum_j exp(scale*S_ij - m_s)
 * o_part : out, fp32 [n_splits][B][H][Nq][d] O_s / l_s; 16-byte aligned
 * 1 <= n_splits <= 65535.
 */
int fa_fwd_partial(const void* q, const void* k, const void* v, float* m_part, float* l_part,
                   float* o_part, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   int n_splits, void* stream);

/*
 * Merge n_splits partial triples per row with the two-block merge rule
 * (airsota.com online-softmax card, section 三, "Running Combined Updates"),
 * in its n-way form (associative: "La recurrencia del online softmax",
 * practice problem 4):
 *   M = max_s m_s;  w_s = l_s exp(m_s - M);  l = sum_s w_s;
 *   O = sum_s w_s O_s / l;  LSE = M + ln l;  l = 0 -> O = 0, LSE = -inf.
 *
 * m_part, l_part : in, fp32 [n_splits][B][H][Nq] (layout of fa_fwd_partial)
 * o_part         : in, fp32 [n_splits][B][H][Nq][d], 16-byte aligned
 * o              : out, bf16 [B][H][Nq][d], 16-byte aligned
 * lse            : out, fp32 [B][H][Nq]
 */
int fa_merge_splits(const float* m_part, const float* l_part, const float* o_part, void* o,
                    float* lse, int B, int H, int Nq, int d, int n_splits, void* stream);

/* Bytes of workspace fa_fwd takes for split-KV with these sizes: m and l
 * fp32, O bf16, each block 256-byte aligned (0 for n_splits <= 1 or invalid
 * sizes). */
size_t fa_split_workspace_bytes(int B, int H, int Nq, int d, int n_splits);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT if any kernel of this library
 * recorded a timed-out wait since the last call, FA_ERR_DEVICE_CHECK (debug
 * build only) if a bounds check failed first, FA_ERR_UNSUPPORTED if a
 * backward kernel found its dynamic shared memory base less than 1024-byte
 * aligned (its layout fills the 227 KB limit and has no room to realign; it
 * then writes nothing), or FA_ERR_CUDA.  The word is
 * one per device, shared by every call on that device (all streams, and the
 * host-buffer entry points, which read it before returning): a timeout from a
 * kernel on another stream is reported to whichever caller reads the word
 * first, and reading clears it.
 */
int fa_get_device_status(void* stream);

/* Static description of an FA_* code; for FA_ERR_CUDA, the text of the last
 * CUDA error seen by this thread.  Never NULL. */
const char* fa_strerror(int code);

/*
 * Split-KV forward that allocates nothing.  No counterpart on the source
 * pages: this is a deployment variant of fa_fwd with n_splits > 1.
 *
 * For callers that cannot allocate device memory on this path: runtimes
 * without a device allocator, hosts whose device memory all belongs to their
 * own pool (a cudaMalloc there would fail or steal from it), and latency-bound
 * loops where an allocation could block or synchronise.  fa_fwd takes its
 * split-KV workspace with cudaMallocAsync; this call puts the same partial
 * (m, l, O) triples in a fixed device array of FA_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until the process exits, then merges
 * them with the same kernels.
 *
 * Arguments and results: as fa_fwd (q, k, v, o, lse, sizes, scale, causal,
 * stream), with 2 <= n_splits <= 65535, clamped to ceil(Nk/128) like fa_fwd;
 * if that leaves one split, the call is fa_fwd with n_splits = 1.
 * The workspace needs about n_splits * B*H*Nq * (2 d + 8) bytes
 * (fa_split_workspace_bytes); a call
 * that needs more than FA_NOALLOC_SCRATCH_BYTES returns
 * FA_ERR_SCRATCH_TOO_SMALL before launching anything.
 *
 * No cudaMalloc, cudaFree or other allocating call is made.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * Like every entry point, the first call with a given head dimension and
 * query-tile count also runs the library's one-time kernel set-up (attribute
 * queries).  All calls share the one array and it keeps the last call's
 * contents: calls that may overlap on the GPU (different streams, or
 * different host threads without ordering) race on it and must be
 * serialised by the caller.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Nq, int Nk, int d, float scale, int causal, int n_splits,
                         void* stream);

/*
 * Softmax over the rows of a matrix with the online normaliser, the two-pass
 * scheme of "Online Softmax 算法详解" section 2.2: pass 1 keeps a running max m
 * and a sum l rescaled by exp(m_old - m_new) whenever the max grows; pass 2
 * writes y = exp(x - m) / l.  Not part of the attention forward: the same
 * recurrence on a plain row operation.
 *
 * x     : in,  [rows][cols] dense row-major, fp32 (dtype FA_DTYPE_F32) or
 *         bf16 (FA_DTYPE_BF16); entries finite or -inf.
 * y     : out, same shape and dtype; may be x (in place).  bf16 results are
 *         the fp32 values rounded to nearest even.
 * lse   : out, fp32 [rows], ln sum_j exp(x_ij) (natural log), or NULL.
 * A row with no finite entry gets y = 0 and lse = -inf.
 * rows >= 0 (0: nothing is launched), 1 <= cols <= 2^30; x and y aligned to
 * their element size (16-byte aligned rows take the vector path).
 * Arithmetic in fp32 with exp as 2^(t log2 e) (ex2.approx): relative error of
 * y about 1e-6 (1 + |x_ij| + |max_j x_ij|), see the tests.
 * Rows up to 16384 fp32 / 32768 bf16 columns run one CTA per row; longer rows
 * a cluster of up to 8 CTAs (up to 131072 fp32 / 262144 bf16 columns held on
 * chip, x read once); longer still, pass 2 reads the row again.
 */
#define FA_DTYPE_F32 0
#define FA_DTYPE_BF16 1
int fa_softmax_rows(const void* x, void* y, float* lse, long long rows, int cols, int dtype,
                    void* stream);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
