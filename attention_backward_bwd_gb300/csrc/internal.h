// Internal parameter blocks and launcher declarations shared by the host API
// (api.cu) and the kernels.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/attn_bwd.h"

namespace attn {

// Query/key tile height of the backward kernels; workspace rows are padded to it.
constexpr int kTileRows = 128;

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ inline int ceil_div(int x, int m) { return (x + m - 1) / m; }

struct SeqParams {
  const int* cu_q;  // nullptr in padded mode
  const int* cu_k;
  int seqlen_q;     // padded: per-sequence length; varlen: total packed rows
  int seqlen_k;
  int batch;        // number of sequences
  const int* used_q = nullptr;  // optional used length of each sequence (<= its rows)
  const int* used_k = nullptr;
};

// A [B, S, H, D] (or packed [total, H, D]) tensor: element strides, last dim contiguous.
struct TensorArg {
  const void* ptr;
  int64_t sb, ss, sh;
};

struct BwdParams {
  SeqParams seq;
  TensorArg q, k, v, o, dout, dq, dk, dv;
  const float* lse;  // natural log, [B, Hq, Sq] or [Hq, total_q]
  // workspace
  float* lse2;   // [Hq][ws_rows]
  float* delta;  // [Hq][ws_rows]
  float* dqacc;  // [Hq][ws_rows][D]
  int* sem;      // [Hq][ws_rows / kTileRows][4]: one per (query tile, 32-row quarter)
  int* sched;    // work counters of the persistent main kernel(s) (after the semaphores)
  int64_t ws_rows;
  int h_q, h_k, head_dim;
  int win_left, win_right;  // local mask sides, -1 = unbounded; causal is (-1, 0)
  int deterministic;
  float scale, scale_log2;
  // logit cap c (0 = off): P = exp2(cap_out * tanh(S * cap_in) - LSE2) with
  // cap_in = scale / c and cap_out = c * log2(e); dS gains the factor 1 - tanh^2
  float softcap, cap_in, cap_out;
  int max_seqlen_q, max_seqlen_k;
  unsigned int* status;
  const unsigned int* input_bad;  // nonzero after cu_seqlens failed validation (varlen)
  unsigned long long timeout_ns;
  // Work-unit order of the KV-stationary kernels, chosen by each kernel's launch:
  // u = outer * unit_per + mid * h_k + g, with (outer, mid) = (b, n) when
  // unit_seq_major, else (n, b); unit_per = the units of one outer index.
  int unit_seq_major, unit_per;
};

struct FwdParams {
  SeqParams seq;
  TensorArg q, k, v, o;
  float* lse;
  int h_q, h_k, head_dim;
  int win_left, win_right;  // local mask sides, -1 = unbounded; causal is (-1, 0)
  float scale_log2;
  float softcap, cap_in, cap_out;  // logit cap as in BwdParams (0 = off)
  int max_seqlen_q;
  const unsigned int* input_bad;
  unsigned int* status;            // device status word (bounded waits that gave up)
  unsigned long long timeout_ns;   // limit of every device-side wait
};

// Workspace layout (byte offsets), identical on host and device.
struct WsLayout {
  int64_t rows;
  size_t off_lse2, off_delta, off_dqacc, off_sem, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The kernels run D = 64, 128 or 256; a head dimension that is a multiple of 8
// below one of those runs on the next with the extra columns zero (TMA's
// out-of-bounds fill on loads, masked stores), and the fp32 dQ accumulator is
// laid out at the padded width.
__host__ __device__ inline int pad_head_dim(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 256); }

// Work counters after the semaphores: one per launch of the persistent
// backward kernels (the D = 256 backward runs two passes).
constexpr int kSchedCounters = 2;

inline WsLayout ws_layout(int batch, int seqlen_q, int h_q, int head_dim, int varlen) {
  WsLayout w;
  if (varlen) {
    w.rows = round_up(seqlen_q + batch * kTileRows, kTileRows);
  } else {
    w.rows = static_cast<int64_t>(batch) * round_up(seqlen_q, kTileRows);
  }
  const size_t per_row = static_cast<size_t>(h_q) * static_cast<size_t>(w.rows);
  w.off_lse2 = 0;
  w.off_delta = align256(w.off_lse2 + per_row * 4);
  w.off_dqacc = align256(w.off_delta + per_row * 4);
  w.off_sem = align256(w.off_dqacc + per_row * static_cast<size_t>(pad_head_dim(head_dim)) * 4);
  // semaphores (one per 32-row quarter of each query tile), then the int32 work
  // counters of the persistent scheduler
  w.total = align256(w.off_sem +
                     (static_cast<size_t>(h_q) * (w.rows / kTileRows) * 4 + kSchedCounters) * 4);
  return w;
}

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_preprocess(const BwdParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_postprocess(const BwdParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdParams& p, int dtype, cudaStream_t stream);
// Head dimensions above 128: the two-pass D = 256 backward (bwd_wide.cu).
cudaError_t launch_bwd_wide(const BwdParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_fwd(const FwdParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_zero_rows(const TensorArg& t, int dtype, int nseq, int rows_per_seq,
                             const int* cu, int total_rows, int heads, int head_dim,
                             cudaStream_t stream);

cudaError_t launch_validate_cu(const int* cu_q, const int* cu_k, int batch, int total_q,
                               int total_k, int max_q, int max_k, unsigned int* bad,
                               cudaStream_t stream);
// Checks 0 <= used[b] <= rows of sequence b for the used-length arrays given.
cudaError_t launch_validate_used(const SeqParams& s, unsigned int* bad, cudaStream_t stream);

int num_sms();

// Device status words of the current device ([0] waits, [1] input validation).
unsigned int* status_word();

// 4-D TMA map over a [B, S, H, D] tensor (dims D, S, H, B; element strides from
// `t`), box {64, box_rows, 1, 1}, 128-byte swizzle, zero fill out of bounds.
// For packed varlen tensors pass batch = 1 and rows = total rows.
bool encode_tmap_bshd(CUtensorMap* out, const TensorArg& t, int dtype, int rows, int heads,
                      int batch, int head_dim, int box_rows);

// 2-D TMA map over a row-major fp32 matrix [rows][cols], box {32, 32}, 128-byte
// swizzle (used to reduce-add dQ tiles into the dQ accumulator).
bool encode_tmap_f32_2d(CUtensorMap* out, float* base, int64_t rows, int cols);

// ---- host side of one backward call (api.cu) ----

// Error message of the calling thread, read back by attn_last_error().
void clear_error();
int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int cuda_fail(cudaError_t e, const char* what);

// Arguments checked and bound to kernel parameters; nothing launched yet.
struct Prepared {
  BwdParams p;
  int dtype;
  bool empty_q, empty_k;
};

int check_common(int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                 int head_dim, float scale, const int* cu_q, const int* cu_k, int max_seqlen_q,
                 int max_seqlen_k);

int prepare_bwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, const float* lse, const attn_tensor* dout,
                const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
                float scale, int causal, const int* cu_q, const int* cu_k, int max_seqlen_q,
                int max_seqlen_k, int deterministic, const attn_opts* opts, void* workspace,
                size_t workspace_bytes, Prepared* out);

// NULL -> no window, no cap; checks the values (ATTN_ERR_ARG).
int resolve_opts(const attn_opts* in, attn_opts* out);

enum Stage { kPre = 1, kMain = 2, kPost = 4 };

// Launches the selected stages (preprocess, main, postprocess) on `stream`.
int run_stages(int stages, const Prepared& pr, cudaStream_t stream);

}  // namespace attn
