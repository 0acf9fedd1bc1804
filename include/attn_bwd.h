/*
 * attn_bwd.h -- C ABI of the GB300 (sm_103a) fused attention backward library
 * (libattn_gb300.so).
 *
 * Problem (TileLang test_tilelang_kernel_mha_bwd.py, ref_program and
 * flashattn_bwd; flash-attention csrc/flash_attn_ck/mha_bwd.cpp, mha_bwd):
 * for every sequence b and query head h, with key/value head g = h / (H_q/H_k)
 * and scale s,
 *     S = s Q K^T (causal: key j allowed for query i iff j <= i + Sk - Sq),
 *     P = softmax(S) = exp(S - LSE),  O = P V,
 *     dV_g = sum over the group of P^T dO,   dP = dO V^T,
 *     Delta = rowsum(O * dO),   dS = P * (dP - Delta),
 *     dQ = s dS K,   dK_g = s * sum over the group of dS^T Q,
 * computed without materialising S or P in memory.
 *
 * Layout.  Q, O, dO, dQ are [B, Sq, H_q, D]; K, V, dK, dV are [B, Sk, H_k, D]
 * (flash-attention mha_bwd argument comments).  Each tensor is passed as an
 * attn_tensor: a device pointer plus element strides for the batch, sequence
 * and head dimensions; the head dimension is contiguous (stride 1).  In varlen
 * mode (cu_seqlens given) tensors are packed [total, H, D], stride_b is
 * ignored, and seqlen_q / seqlen_k are the TOTAL packed row counts while
 * max_seqlen_q / max_seqlen_k bound the per-sequence lengths.  cu_seqlens_q
 * and cu_seqlens_k may differ (cross attention: sequence b has
 * cu_q[b+1]-cu_q[b] queries and cu_k[b+1]-cu_k[b] keys, causal masks aligned
 * bottom-right per sequence); a sequence with keys but no queries gets
 * dK = dV = 0, one with queries but no keys dQ = 0.
 * LSE is fp32, natural log: [B, H_q, Sq] contiguous, or [H_q, total_q] in
 * varlen mode (flash-attention's softmax_lse).
 *
 * Supported: dtype fp16 or bf16 (all of Q,K,V,O,dO,dQ,dK,dV share it), D a
 * multiple of 8 in [8, 256] (the head sizes the CK wrapper's mha_bwd accepts;
 * 64, 96, 128, 192 and 256 run natively (96 without a logit cap or a left
 * window side), any other D runs on the next of those with the extra
 * head-dimension columns zero; above 128 the backward runs as two passes, one
 * for dV and one for dK and dQ), H_q % H_k == 0, base pointers and
 * strides 16-byte aligned (strides multiples of 8 elements).
 *
 * Ownership.  The caller owns every buffer, including the workspace; the
 * library allocates nothing per call and keeps no state across calls except
 * one-time kernel attributes, a device status word and, once attn_bwd_host
 * has been called on a device, that call's internal streams and events.  All compute calls
 * are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *
 * Errors.  Every call returns ATTN_OK (0) or a negative code and then
 * attn_last_error() gives a message (thread-local).  Argument errors are
 * detected on the host before anything is launched (the convention of
 * mha_bwd's argument checks: a negative return means invalid argument).
 * Device-side waits are bounded; a wait that gives up records a nonzero
 * status that attn_check_device_status() reports as ATTN_ERR_DEVICE_TIMEOUT.
 */
#ifndef ATTN_BWD_GB300_H
#define ATTN_BWD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same type as cudaStream_t */

enum attn_dtype { ATTN_FP16 = 0, ATTN_BF16 = 1 };

enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_DTYPE = -1,          /* dtype not fp16/bf16 */
  ATTN_ERR_SHAPE = -2,          /* bad sizes: B<=0, H_q%H_k, D not 8..256 by 8 */
  ATTN_ERR_STRIDE = -3,         /* stride not a multiple of 8 elements or negative */
  ATTN_ERR_ALIGN = -4,          /* base pointer not 16-byte aligned */
  ATTN_ERR_NULL = -5,           /* required pointer is NULL */
  ATTN_ERR_WORKSPACE = -6,      /* workspace missing, misaligned or too small */
  ATTN_ERR_CUDA = -7,           /* a CUDA launch or runtime call failed */
  ATTN_ERR_DEVICE_TIMEOUT = -8, /* a bounded device wait gave up */
  ATTN_ERR_ARG = -9             /* other invalid argument (scale, max_seqlen, ...) */
};

typedef struct {
  void* ptr;        /* device pointer to element [0,0,0,0] */
  int64_t stride_b; /* elements between batches (ignored in varlen mode) */
  int64_t stride_s; /* elements between sequence positions */
  int64_t stride_h; /* elements between heads; the D dimension has stride 1 */
} attn_tensor;

/*
 * attn_fwd -- forward pass producing O and the natural-log LSE that
 * attn_bwd consumes (TileLang flashattn_fwd, online softmax).  Supporting
 * call: the library's subject is the backward.  Rows with no allowed key get
 * O = 0 and LSE = +inf.  q, k, v are read; o and lse are written.
 */
int attn_fwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
             const attn_tensor* o, float* lse, int dtype, int batch, int seqlen_q,
             int seqlen_k, int h_q, int h_k, int head_dim, float scale, int causal,
             const int* cu_seqlens_q, const int* cu_seqlens_k, int max_seqlen_q,
             int max_seqlen_k, attn_stream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs
 * (flash-attention hopper/flash_bwd_launch_template.h, run_flash_bwd:
 * softmax_lse_log2, dsoftmax_sum, dq_accum and dq_semaphore).
 * varlen != 0: seqlen_q is the total packed query rows and batch the number
 * of sequences.  Workspace rows are padded to 128 per sequence.
 */
size_t attn_bwd_workspace_size(int batch, int seqlen_q, int h_q, int head_dim,
                               int deterministic, int varlen);

/*
 * attn_bwd_workspace_layout -- where the pieces of the workspace live, for
 * callers that inspect them.  Writes byte offsets of LSE2 (fp32
 * [H_q][rows]), Delta (fp32 [H_q][rows]), dQaccum (fp32 [H_q][rows][D]) and
 * the semaphores (int32 [H_q][rows/128][4], one per 32-row quarter of a
 * query tile, followed by two int32 work counters of the main kernels'
 * schedulers) into offsets[0..3], and `rows`.  dQaccum's
 * row width D is the head dimension padded to 64, 128 or 256.
 * Row of query i of sequence b: padded mode b*round_up(Sq,128) + i; varlen
 * 128*(cu_seqlens_q[b]/128 + b) + i.  Returns ATTN_OK or ATTN_ERR_NULL.
 */
int attn_bwd_workspace_layout(int batch, int seqlen_q, int h_q, int head_dim, int varlen,
                              size_t offsets[4], int64_t* rows);

/*
 * attn_bwd -- fused backward: dq, dk, dv from q, k, v, o, lse, dout.
 * Runs the three stages below on `stream`.  dq, dk, dv are fully overwritten.
 * deterministic != 0: dQ contributions are added in ascending key-tile order,
 * so results are bit-identical run to run (in the reference CK wrapper the
 * same property comes from split dq_accum buffers; here a semaphore orders
 * the adds).  Sq == 0 gives dk = dv = 0; Sk == 0 gives dq = 0.
 * workspace: device memory of at least attn_bwd_workspace_size(...) bytes,
 * 256-byte aligned, owned by the caller, not shared by concurrent calls.
 */
int attn_bwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
             const attn_tensor* o, const float* lse, const attn_tensor* dout,
             const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
             int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
             float scale, int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
             int max_seqlen_q, int max_seqlen_k, int deterministic, void* workspace,
             size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_opts -- optional mask and logit settings of attn_fwd_ex / attn_bwd_ex
 * (NULL = no window, no cap: the behaviour of attn_fwd / attn_bwd).  Note
 * that a zeroed struct is NOT that default: window (0, 0) lets each query see
 * one key.
 *   window_left, window_right: a local (sliding-window) mask, the window of
 *     flash-attention csrc/flash_attn_ck/mha_bwd.cpp (mha_bwd's mask set-up),
 *     -1 meaning unbounded on that side.  Bottom-right aligned like causal:
 *     with off = Sk - Sq (per sequence in varlen mode), query i attends key j
 *     iff j >= i + off - window_left (when window_left >= 0) and
 *     j <= i + off + window_right (when window_right >= 0).  causal != 0 sets
 *     window_right to 0, so (window_left = W, causal = 1) is sliding-window
 *     causal attention.  Rows that see no key get O = 0, LSE = +inf, dQ = 0;
 *     keys that no query sees get dK = dV = 0.
 *   softcap: > 0 caps the logits s = scale * q.k as softcap * tanh(s / softcap)
 *     before the softmax (the Has_softcap path of flash-attention
 *     hopper/flash_bwd_launch_template.h; the formula is the usual logit cap);
 *     the backward applies the cap's derivative.  0 = no cap.
 *   seqused_q, seqused_k: NULL, or device int32 arrays [batch]: sequence b
 *     is the first seqused[b] of its rows (its padded slab, or its packed
 *     range from cu_seqlens), the seqused_q / seqused_k of the FA3 launcher
 *     (flash-attention hopper/flash_bwd_launch_template.h).  The other rows of
 *     the sequence take no part in the result and their dq / dk / dv rows (O
 *     and LSE rows in the forward) are left as they were.  Like the packed
 *     rows of a neighbouring sequence, they may be read inside a tile and
 *     masked out, so they must hold finite values (0 x NaN is NaN in a tensor
 *     core sum).  Values outside [0, rows of the sequence] are reported by
 *     attn_check_device_status as ATTN_ERR_ARG and make the kernels return.
 * Window sides below -1, a negative or non-finite softcap give ATTN_ERR_ARG.
 */
typedef struct {
  int window_left;
  int window_right;
  float softcap;
  const int* seqused_q;
  const int* seqused_k;
} attn_opts;

/*
 * attn_bwd_ex -- attn_bwd with attn_opts, running the stages selected by the
 * bit mask `stages` (1 = preprocess, 2 = main, 4 = postprocess; 7 = all, in
 * that order; outside 1..7: ATTN_ERR_ARG).  The stages of one backward must
 * share the workspace and the options.  Deterministic mode orders the dQ adds
 * of each query tile over the key tiles that see it.
 * attn_fwd_ex -- attn_fwd with attn_opts (produces the O and LSE that
 * attn_bwd_ex with the same options consumes).
 */
int attn_bwd_ex(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, const float* lse, const attn_tensor* dout,
                const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim, float scale,
                int causal, const int* cu_seqlens_q, const int* cu_seqlens_k, int max_seqlen_q,
                int max_seqlen_k, int deterministic, const attn_opts* opts, int stages,
                void* workspace, size_t workspace_bytes, attn_stream_t stream);
int attn_fwd_ex(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, float* lse, int dtype, int batch, int seqlen_q, int seqlen_k,
                int h_q, int h_k, int head_dim, float scale, int causal, const int* cu_seqlens_q,
                const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                const attn_opts* opts, attn_stream_t stream);

/*
 * attn_bwd_noalloc -- attn_bwd with no workspace argument, for callers that
 * must not allocate device memory: code whose device memory all belongs to
 * another allocator (a framework's memory pool or an arena reserved at
 * start-up), where a cudaMalloc in the middle of a step would either fail
 * because the arena already holds the memory or stall the device while the
 * driver allocates.  The pages describe no counterpart of this call.
 *
 * Arguments and results are those of attn_bwd minus workspace and
 * workspace_bytes; it allocates nothing.  Its workspace is a static array of
 * 32 MiB in device memory inside the library, which every GPU that loads the
 * library keeps until the process exits.  A problem whose
 * attn_bwd_workspace_size(...) exceeds 32 MiB is rejected with
 * ATTN_ERR_WORKSPACE and a message (use attn_bwd then); 32 MiB covers, for
 * example, B*H_q*round_up(Sq,128) up to about 1.2e5 query rows at D = 64.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Each call clears what must start at zero.
 * All calls on a device share the one array: calls that overlap on the GPU
 * (other streams, other host threads) race and corrupt each other's results,
 * so issue them one after another on one stream.
 */
int attn_bwd_noalloc(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                     const attn_tensor* o, const float* lse, const attn_tensor* dout,
                     const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv,
                     int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                     int head_dim, float scale, int causal, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                     int deterministic, attn_stream_t stream);

/*
 * attn_bwd_host -- attn_bwd on tensors in HOST memory: copies q, k, v, o,
 * dout and lse to the device, runs the backward, and copies dq, dk, dv back,
 * all enqueued on `stream` (the call returns before the work is done; the
 * results are in host memory once `stream` has passed this call, e.g. after
 * cudaStreamSynchronize).  The pages describe no counterpart of this call:
 * it serves callers whose activations live in host memory (offloaded
 * activations), where the copies would otherwise cost more than the kernels.
 *
 * The problem is cut into `chunks` independent pieces (0 = the library
 * chooses, currently 8; at most 64): runs of whole sequences when batch >=
 * chunks, else one sequence and a range of key/value heads with their query
 * heads.  Each piece's copies in, kernels and copies out run on internal
 * streams, so the copies of one piece overlap the kernels of the others.
 * Results equal attn_bwd's on the same data (bit for bit in deterministic
 * mode and for dK, dV; dQ's fp32 adds may be ordered differently otherwise).
 *
 * Host tensors: padded [B, S, H, D] (no varlen), the heads of a position
 * adjacent (stride_h == D), D contiguous, and positions and sequences not
 * overlapping; lse is [B, H_q, Sq] contiguous.  Page-locked memory
 * (cudaHostAlloc / cudaHostRegister) is needed for the copies to overlap;
 * pageable memory works but serialises them.
 * device_buffer: device memory of at least
 * attn_bwd_host_buffer_size(batch, seqlen_q, seqlen_k, h_q, h_k, head_dim,
 * chunks) bytes, 256-byte aligned, owned by the caller, not used by any other
 * call while this one runs.  It holds device copies of all eight tensors and
 * of lse plus three chunk-sized workspaces (one per internal compute stream).
 * opts: a local window and a logit cap as for attn_bwd_ex (NULL: none);
 * seqused_q/k must be NULL here (ATTN_ERR_ARG otherwise).
 * Errors as attn_bwd (argument errors before anything is enqueued; a
 * stride_h other than D is ATTN_ERR_STRIDE).  The first call on a device
 * creates the library's internal streams and events for that device; make
 * it before any stream capture.
 */
size_t attn_bwd_host_buffer_size(int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                                 int head_dim, int chunks);
int attn_bwd_host(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                  const attn_tensor* o, const float* lse, const attn_tensor* dout,
                  const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                  int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
                  float scale, int causal, int deterministic, const attn_opts* opts, int chunks,
                  void* device_buffer, size_t device_buffer_bytes, attn_stream_t stream);

/*
 * attn_bwd_host_varlen -- attn_bwd_host for packed [total, H, D] tensors with
 * cu_seqlens_q / cu_seqlens_k in HOST memory (int32 [batch + 1], starting at
 * 0, nondecreasing, ending at total_q / total_k; checked on the host:
 * ATTN_ERR_ARG).  A chunk is a run of whole sequences holding about an equal
 * share of the attention work; each tensor's rows of a chunk move in one
 * pitched copy.  lse is [H_q, total_q] in host memory.  Host tensors need
 * adjacent heads (stride_h == D) and stride_s >= H * D.  device_buffer: at
 * least attn_bwd_host_varlen_buffer_size(...) bytes (0 means invalid
 * arguments or cu_seqlens).  Everything else as attn_bwd_host.
 */
size_t attn_bwd_host_varlen_buffer_size(const int* cu_seqlens_q, const int* cu_seqlens_k,
                                        int batch, int total_q, int total_k, int h_q, int h_k,
                                        int head_dim, int chunks);
int attn_bwd_host_varlen(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                         const attn_tensor* o, const float* lse, const attn_tensor* dout,
                         const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv,
                         int dtype, int batch, int total_q, int total_k, int h_q, int h_k,
                         int head_dim, float scale, int causal, const int* cu_seqlens_q,
                         const int* cu_seqlens_k, int deterministic, const attn_opts* opts,
                         int chunks, void* device_buffer, size_t device_buffer_bytes,
                         attn_stream_t stream);

/*
 * The three stages of attn_bwd, callable one by one (same arguments, same
 * checks) so that each kernel can be timed on its own.  They must run in this
 * order on one stream with the same workspace.
 *   attn_bwd_preprocess  -- Delta = rowsum(O*dO) (fp32), LSE2 = LSE*log2(e),
 *                           dQaccum = 0, semaphores = 0
 *                           (TileLang flashattn_bwd_preprocess; FA3 preprocess
 *                           with Clear_dQaccum).
 *   attn_bwd_main        -- dK, dV written; dQ accumulated in fp32 dQaccum
 *                           (TileLang flashattn_bwd; FA3 CollectiveMainloopBwd).
 *   attn_bwd_postprocess -- dQ = scale * dQaccum cast to the dtype
 *                           (mslk flash_bwd_postprocess.py; FA3
 *                           FlashAttnBwdPostprocessConvertdQ).
 */
int attn_bwd_preprocess(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                        const attn_tensor* o, const float* lse, const attn_tensor* dout,
                        const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv,
                        int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                        int head_dim, float scale, int causal, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                        int deterministic, void* workspace, size_t workspace_bytes,
                        attn_stream_t stream);
int attn_bwd_main(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                  const attn_tensor* o, const float* lse, const attn_tensor* dout,
                  const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                  int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
                  float scale, int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  int max_seqlen_q, int max_seqlen_k, int deterministic, void* workspace,
                  size_t workspace_bytes, attn_stream_t stream);
int attn_bwd_postprocess(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                         const attn_tensor* o, const float* lse, const attn_tensor* dout,
                         const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv,
                         int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                         int head_dim, float scale, int causal, const int* cu_seqlens_q,
                         const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                         int deterministic, void* workspace, size_t workspace_bytes,
                         attn_stream_t stream);

/*
 * attn_check_device_status -- synchronises `stream`, then reads and clears the
 * device status word.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (a bounded
 * wait inside a kernel gave up; attn_last_error names the wait site),
 * ATTN_ERR_ARG (cu_seqlens or seqused_q/k failed the device-side check;
 * attn_last_error names which) or ATTN_ERR_CUDA (the stream reported an error).
 * The status word is one per device and stays set until this call clears it.
 * While a failed cu_seqlens / seqused check is recorded there, the kernels of
 * EVERY later varlen or seqused call on that device (any stream, any host
 * thread, valid arrays or not) return at once without writing their outputs,
 * and those calls still return ATTN_OK on the host.  A caller that passes
 * device offsets it has not validated itself should therefore call this
 * function after such a call, before relying on any later varlen result.
 */
int attn_check_device_status(attn_stream_t stream);

/*
 * attn_set_wait_timeout_ns -- limit for every device-side wait of later calls
 * (default 4e9 ns).  Values <= 0 restore the default.
 */
void attn_set_wait_timeout_ns(int64_t ns);

/* Message for the last error on this thread ("" if none). */
const char* attn_last_error(void);

/* Library version string. */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_GB300_H */
