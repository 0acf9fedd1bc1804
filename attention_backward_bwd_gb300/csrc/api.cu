// Host implementation of the C ABI declared in include/attn_bwd.h: argument
// checks, workspace layout, TMA descriptor encoding, kernel launch order.
//
// The launch order follows flash-attention hopper/flash_bwd_launch_template.h
// (run_flash_bwd): preprocess -> main -> dQ postprocess, all on the caller's
// stream.  The argument checks follow the guards of flash-attention
// csrc/flash_attn_ck/mha_bwd.cpp (mha_bwd): fp16/bf16 only, contiguous last
// dimension, H_q divisible by H_k, and an empty query side gives zero dK, dV.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/attn_bwd.h"
#include "internal.h"

namespace attn {

namespace {

thread_local std::string g_err;
std::atomic<long long> g_timeout_ns{4000000000LL};

}  // namespace

void clear_error() { g_err.clear(); }

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device status words: [0] = 0 or the site of a bounded wait that gave up;
// [1] = 0 or the code of a failed cu_seqlens validation.
__device__ unsigned int g_device_status[2] = {0u, 0u};

namespace {
constexpr int kMaxDevices = 64;
}  // namespace

unsigned int* status_word() {
  static unsigned int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int num_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

bool encode_tmap_bshd(CUtensorMap* out, const TensorArg& t, int dtype, int rows, int heads,
                      int batch, int head_dim, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows <= 0 || heads <= 0 || batch <= 0) return false;
  const cuuint64_t esz = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  // byte strides of dims 1..3; with a single batch the batch stride is never
  // used, but the map still needs a valid (16-byte multiple) value
  const int64_t sb = batch > 1 ? t.sb : t.ss * static_cast<int64_t>(rows);
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(t.ss) * esz, static_cast<cuuint64_t>(t.sh) * esz,
                           static_cast<cuuint64_t>(sb) * esz};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(out,
                        dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(t.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_f32_2d(CUtensorMap* out, float* base, int64_t rows, int cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows <= 0 || cols <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

int check_tensor(const attn_tensor* t, const char* name, bool varlen, bool need) {
  if (t == nullptr) return fail(ATTN_ERR_NULL, "%s: descriptor is NULL", name);
  if (!need) return ATTN_OK;
  if (t->ptr == nullptr) return fail(ATTN_ERR_NULL, "%s: pointer is NULL", name);
  if (reinterpret_cast<uintptr_t>(t->ptr) % 16 != 0)
    return fail(ATTN_ERR_ALIGN, "%s: base pointer must be 16-byte aligned", name);
  const int64_t st[3] = {t->stride_b, t->stride_s, t->stride_h};
  for (int i = varlen ? 1 : 0; i < 3; ++i) {
    if (st[i] <= 0 || st[i] % 8 != 0)
      return fail(ATTN_ERR_STRIDE,
                  "%s: strides must be positive multiples of 8 elements (got b=%lld s=%lld h=%lld)",
                  name, static_cast<long long>(t->stride_b), static_cast<long long>(t->stride_s),
                  static_cast<long long>(t->stride_h));
  }
  return ATTN_OK;
}

TensorArg targ(const attn_tensor* t) {
  return TensorArg{t->ptr, t->stride_b, t->stride_s, t->stride_h};
}

}  // namespace

int check_common(int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                 int head_dim, float scale, const int* cu_q, const int* cu_k,
                 int max_seqlen_q, int max_seqlen_k) {
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_DTYPE, "dtype must be ATTN_FP16 (0) or ATTN_BF16 (1), got %d", dtype);
  if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0)
    return fail(ATTN_ERR_SHAPE, "head_dim must be a multiple of 8 in [8, 256], got %d", head_dim);
  if (batch <= 0) return fail(ATTN_ERR_SHAPE, "batch must be positive, got %d", batch);
  if (h_q <= 0 || h_k <= 0 || h_q % h_k != 0)
    return fail(ATTN_ERR_SHAPE, "h_q (%d) must be a positive multiple of h_k (%d)", h_q, h_k);
  if (seqlen_q < 0 || seqlen_k < 0)
    return fail(ATTN_ERR_SHAPE, "sequence lengths must be >= 0 (got %d, %d)", seqlen_q, seqlen_k);
  if (!std::isfinite(scale)) return fail(ATTN_ERR_ARG, "scale must be finite");
  if ((cu_q == nullptr) != (cu_k == nullptr))
    return fail(ATTN_ERR_ARG, "cu_seqlens_q and cu_seqlens_k must both be given or both be NULL");
  if (cu_q != nullptr) {
    if (max_seqlen_q < 0 || max_seqlen_k < 0 || max_seqlen_q > seqlen_q ||
        max_seqlen_k > seqlen_k)
      return fail(ATTN_ERR_ARG,
                  "varlen: max_seqlen_q/k (%d, %d) must lie in [0, total rows (%d, %d)]",
                  max_seqlen_q, max_seqlen_k, seqlen_q, seqlen_k);
  }
  return ATTN_OK;
}

int resolve_opts(const attn_opts* in, attn_opts* out) {
  *out = attn_opts{-1, -1, 0.f, nullptr, nullptr};
  if (in == nullptr) return ATTN_OK;
  if (in->window_left < -1 || in->window_right < -1)
    return fail(ATTN_ERR_ARG, "window sides must be >= -1 (-1 = unbounded), got (%d, %d)",
                in->window_left, in->window_right);
  if (!std::isfinite(in->softcap) || in->softcap < 0.f)
    return fail(ATTN_ERR_ARG, "softcap must be finite and >= 0 (0 = off), got %g",
                static_cast<double>(in->softcap));
  *out = *in;
  return ATTN_OK;
}

int prepare_bwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, const float* lse, const attn_tensor* dout,
                const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
                float scale, int causal, const int* cu_q, const int* cu_k, int max_seqlen_q,
                int max_seqlen_k, int deterministic, const attn_opts* opts_in, void* workspace,
                size_t workspace_bytes, Prepared* out) {
  int rc = check_common(dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, scale, cu_q, cu_k,
                        max_seqlen_q, max_seqlen_k);
  if (rc) return rc;
  attn_opts opts;
  if ((rc = resolve_opts(opts_in, &opts))) return rc;
  const bool varlen = cu_q != nullptr;
  const bool hq = seqlen_q > 0, hk = seqlen_k > 0;
  if ((rc = check_tensor(q, "q", varlen, hq && hk))) return rc;
  if ((rc = check_tensor(k, "k", varlen, hq && hk))) return rc;
  if ((rc = check_tensor(v, "v", varlen, hq && hk))) return rc;
  if ((rc = check_tensor(o, "o", varlen, hq && hk))) return rc;
  if ((rc = check_tensor(dout, "dout", varlen, hq && hk))) return rc;
  if ((rc = check_tensor(dq, "dq", varlen, hq))) return rc;
  if ((rc = check_tensor(dk, "dk", varlen, hk))) return rc;
  if ((rc = check_tensor(dv, "dv", varlen, hk))) return rc;
  if (hq && hk && lse == nullptr) return fail(ATTN_ERR_NULL, "lse is NULL");
  if (hq && hk && reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(ATTN_ERR_ALIGN, "lse must be 4-byte aligned");
  const WsLayout w = ws_layout(batch, seqlen_q, h_q, head_dim, varlen ? 1 : 0);
  // the dQ accumulator's rows of all heads are one TMA dimension (32-bit coordinates)
  if (w.rows * h_q > INT32_MAX)
    return fail(ATTN_ERR_SHAPE, "too many query rows: %lld accumulator rows x %d heads >= 2^31",
                static_cast<long long>(w.rows), h_q);
  if (hq && hk) {
    if (workspace == nullptr) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
      return fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < w.total)
      return fail(ATTN_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed",
                  workspace_bytes, w.total);
  }
  BwdParams& p = out->p;
  std::memset(&p, 0, sizeof(p));
  p.seq = SeqParams{cu_q, cu_k, seqlen_q, seqlen_k, batch};
  p.q = targ(q);
  p.k = targ(k);
  p.v = targ(v);
  p.o = targ(o);
  p.dout = targ(dout);
  p.dq = targ(dq);
  p.dk = targ(dk);
  p.dv = targ(dv);
  p.lse = lse;
  char* ws = static_cast<char*>(workspace);
  p.lse2 = reinterpret_cast<float*>(ws + w.off_lse2);
  p.delta = reinterpret_cast<float*>(ws + w.off_delta);
  p.dqacc = reinterpret_cast<float*>(ws + w.off_dqacc);
  p.sem = reinterpret_cast<int*>(ws + w.off_sem);
  p.sched = p.sem + static_cast<int64_t>(h_q) * (w.rows / kTileRows) * 4;
  p.ws_rows = w.rows;
  p.h_q = h_q;
  p.h_k = h_k;
  p.head_dim = head_dim;
  p.win_left = opts.window_left;
  p.win_right = causal ? 0 : opts.window_right;  // causal bounds the right side at 0
  p.softcap = opts.softcap;
  p.cap_in = opts.softcap > 0.f ? scale / opts.softcap : 0.f;
  p.cap_out = opts.softcap * 1.4426950408889634f;
  p.deterministic = deterministic ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.max_seqlen_q = varlen ? max_seqlen_q : seqlen_q;
  p.max_seqlen_k = varlen ? max_seqlen_k : seqlen_k;
  p.status = status_word();
  if (p.status == nullptr) return fail(ATTN_ERR_CUDA, "cannot resolve the device status word");
  p.seq.used_q = opts.seqused_q;
  p.seq.used_k = opts.seqused_k;
  const bool used = opts.seqused_q != nullptr || opts.seqused_k != nullptr;
  p.input_bad = (varlen || used) ? p.status + 1 : nullptr;
  p.timeout_ns = static_cast<unsigned long long>(g_timeout_ns.load());
  out->dtype = dtype;
  out->empty_q = !hq;
  out->empty_k = !hk;
  return ATTN_OK;
}

int run_stages(int stages, const Prepared& pr, cudaStream_t stream) {
  const BwdParams& p = pr.p;
  cudaError_t e;
  if (p.seq.cu_q != nullptr && !(pr.empty_q || pr.empty_k)) {
    e = launch_validate_cu(p.seq.cu_q, p.seq.cu_k, p.seq.batch, p.seq.seqlen_q, p.seq.seqlen_k,
                           p.max_seqlen_q, p.max_seqlen_k, p.status + 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cu_seqlens validation launch");
  }
  if ((p.seq.used_q != nullptr || p.seq.used_k != nullptr) && !(pr.empty_q || pr.empty_k)) {
    e = launch_validate_used(p.seq, p.status + 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "seqused validation launch");
  }
  if (pr.empty_q || pr.empty_k) {
    // Nothing to reduce.  Empty query side: dK = dV = 0.  Empty key side: dQ = 0.
    if (stages & kMain) {
      if (pr.empty_q && !pr.empty_k) {
        const int rows_k = p.seq.cu_q ? 0 : p.seq.seqlen_k;
        e = launch_zero_rows(p.dk, pr.dtype, p.seq.batch, rows_k, p.seq.cu_k, p.seq.seqlen_k,
                             p.h_k, p.head_dim, stream);
        if (e != cudaSuccess) return cuda_fail(e, "zero dk");
        e = launch_zero_rows(p.dv, pr.dtype, p.seq.batch, rows_k, p.seq.cu_k, p.seq.seqlen_k,
                             p.h_k, p.head_dim, stream);
        if (e != cudaSuccess) return cuda_fail(e, "zero dv");
      }
    }
    if ((stages & kPost) && pr.empty_k && !pr.empty_q) {
      const int rows_q = p.seq.cu_q ? 0 : p.seq.seqlen_q;
      e = launch_zero_rows(p.dq, pr.dtype, p.seq.batch, rows_q, p.seq.cu_q, p.seq.seqlen_q, p.h_q,
                           p.head_dim, stream);
      if (e != cudaSuccess) return cuda_fail(e, "zero dq");
    }
    return ATTN_OK;
  }
  if (stages & kPre) {
    e = launch_preprocess(p, pr.dtype, stream);
    if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
  }
  if (stages & kMain) {
    e = pad_head_dim(p.head_dim) > 128 ? launch_bwd_wide(p, pr.dtype, stream)
                                       : launch_bwd_main(p, pr.dtype, stream);
    if (e == cudaErrorInvalidValue)
      return fail(ATTN_ERR_CUDA, "main kernel: TMA descriptor encoding or launch failed");
    if (e != cudaSuccess) return cuda_fail(e, "main kernel launch");
  }
  if (stages & kPost) {
    e = launch_postprocess(p, pr.dtype, stream);
    if (e != cudaSuccess) return cuda_fail(e, "postprocess launch");
  }
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

#define ATTN_BWD_ARGS_DECL                                                                   \
  const attn_tensor *q, const attn_tensor *k, const attn_tensor *v, const attn_tensor *o,     \
      const float *lse, const attn_tensor *dout, const attn_tensor *dq, const attn_tensor *dk, \
      const attn_tensor *dv, int dtype, int batch, int seqlen_q, int seqlen_k, int h_q,        \
      int h_k, int head_dim, float scale, int causal, const int *cu_seqlens_q,                 \
      const int *cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, int deterministic,          \
      void *workspace, size_t workspace_bytes, attn_stream_t stream
#define ATTN_BWD_ARGS_PASS                                                                  \
  q, k, v, o, lse, dout, dq, dk, dv, dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, \
      scale, causal, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, deterministic, \
      workspace, workspace_bytes

static int bwd_entry_opts(int stages, const attn_opts* opts, ATTN_BWD_ARGS_DECL) {
  g_err.clear();
  Prepared pr;
  const int rc = prepare_bwd(q, k, v, o, lse, dout, dq, dk, dv, dtype, batch, seqlen_q, seqlen_k,
                             h_q, h_k, head_dim, scale, causal, cu_seqlens_q, cu_seqlens_k,
                             max_seqlen_q, max_seqlen_k, deterministic, opts, workspace,
                             workspace_bytes, &pr);
  if (rc) return rc;
  return run_stages(stages, pr, reinterpret_cast<cudaStream_t>(stream));
}

static int bwd_entry(int stages, ATTN_BWD_ARGS_DECL) {
  return bwd_entry_opts(stages, nullptr, ATTN_BWD_ARGS_PASS, stream);
}

extern "C" {

int attn_bwd(ATTN_BWD_ARGS_DECL) { return bwd_entry(kPre | kMain | kPost, ATTN_BWD_ARGS_PASS, stream); }
int attn_bwd_preprocess(ATTN_BWD_ARGS_DECL) { return bwd_entry(kPre, ATTN_BWD_ARGS_PASS, stream); }
int attn_bwd_main(ATTN_BWD_ARGS_DECL) { return bwd_entry(kMain, ATTN_BWD_ARGS_PASS, stream); }
int attn_bwd_postprocess(ATTN_BWD_ARGS_DECL) {
  return bwd_entry(kPost, ATTN_BWD_ARGS_PASS, stream);
}

int attn_bwd_ex(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, const float* lse, const attn_tensor* dout,
                const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv, int dtype,
                int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim, float scale,
                int causal, const int* cu_seqlens_q, const int* cu_seqlens_k, int max_seqlen_q,
                int max_seqlen_k, int deterministic, const attn_opts* opts, int stages,
                void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (stages <= 0 || stages > (kPre | kMain | kPost)) {
    g_err.clear();
    return fail(ATTN_ERR_ARG, "stages must be a nonzero mask of 1, 2 and 4, got %d", stages);
  }
  return bwd_entry_opts(stages, opts, ATTN_BWD_ARGS_PASS, stream);
}

size_t attn_bwd_workspace_size(int batch, int seqlen_q, int h_q, int head_dim, int deterministic,
                               int varlen) {
  (void)deterministic;  // the semaphores are always part of the layout
  if (batch <= 0 || seqlen_q < 0 || h_q <= 0 || head_dim <= 0) return 0;
  return ws_layout(batch, seqlen_q, h_q, head_dim, varlen).total;
}

int attn_bwd_workspace_layout(int batch, int seqlen_q, int h_q, int head_dim, int varlen,
                              size_t offsets[4], int64_t* rows) {
  if (offsets == nullptr || rows == nullptr) return fail(ATTN_ERR_NULL, "NULL output pointer");
  const WsLayout w = ws_layout(batch, seqlen_q, h_q, head_dim, varlen);
  offsets[0] = w.off_lse2;
  offsets[1] = w.off_delta;
  offsets[2] = w.off_dqacc;
  offsets[3] = w.off_sem;
  *rows = w.rows;
  return ATTN_OK;
}

int attn_fwd_ex(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                const attn_tensor* o, float* lse, int dtype, int batch, int seqlen_q, int seqlen_k,
                int h_q, int h_k, int head_dim, float scale, int causal, const int* cu_seqlens_q,
                const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                const attn_opts* opts_in, attn_stream_t stream) {
  g_err.clear();
  int rc = check_common(dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, scale,
                        cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k);
  if (rc) return rc;
  attn_opts opts;
  if ((rc = resolve_opts(opts_in, &opts))) return rc;
  const bool varlen = cu_seqlens_q != nullptr;
  if (seqlen_q == 0) return ATTN_OK;
  if ((rc = check_tensor(q, "q", varlen, true))) return rc;
  if ((rc = check_tensor(k, "k", varlen, seqlen_k > 0))) return rc;
  if ((rc = check_tensor(v, "v", varlen, seqlen_k > 0))) return rc;
  if ((rc = check_tensor(o, "o", varlen, true))) return rc;
  if (lse == nullptr) return fail(ATTN_ERR_NULL, "lse is NULL");
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.seq = SeqParams{cu_seqlens_q, cu_seqlens_k, seqlen_q, seqlen_k, batch};
  p.seq.used_q = opts.seqused_q;
  p.seq.used_k = opts.seqused_k;
  p.q = targ(q);
  p.k = targ(k);
  p.v = targ(v);
  p.o = targ(o);
  p.lse = lse;
  p.h_q = h_q;
  p.h_k = h_k;
  p.head_dim = head_dim;
  p.win_left = opts.window_left;
  p.win_right = causal ? 0 : opts.window_right;  // causal bounds the right side at 0
  p.softcap = opts.softcap;
  p.cap_in = opts.softcap > 0.f ? scale / opts.softcap : 0.f;
  p.cap_out = opts.softcap * 1.4426950408889634f;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.max_seqlen_q = varlen ? max_seqlen_q : seqlen_q;
  if (p.max_seqlen_q == 0) return ATTN_OK;
  unsigned int* st = status_word();
  if (st == nullptr) return fail(ATTN_ERR_CUDA, "cannot resolve the device status word");
  p.status = st;
  p.timeout_ns = static_cast<unsigned long long>(g_timeout_ns.load());
  cudaError_t e;
  if (varlen) {
    p.input_bad = st + 1;
    e = launch_validate_cu(cu_seqlens_q, cu_seqlens_k, batch, seqlen_q, seqlen_k, max_seqlen_q,
                           max_seqlen_k, st + 1, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cu_seqlens validation launch");
  }
  if (p.seq.used_q != nullptr || p.seq.used_k != nullptr) {
    p.input_bad = st + 1;
    e = launch_validate_used(p.seq, st + 1, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "seqused validation launch");
  }
  e = launch_fwd(p, dtype, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ATTN_OK;
}

int attn_fwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
             const attn_tensor* o, float* lse, int dtype, int batch, int seqlen_q, int seqlen_k,
             int h_q, int h_k, int head_dim, float scale, int causal, const int* cu_seqlens_q,
             const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, attn_stream_t stream) {
  return attn_fwd_ex(q, k, v, o, lse, dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim,
                     scale, causal, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                     nullptr, stream);
}

int attn_check_device_status(attn_stream_t stream) {
  g_err.clear();
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int v[2] = {0u, 0u};
  e = cudaMemcpyFromSymbol(v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  if (v[0] != 0 || v[1] != 0) {
    const unsigned int zero[2] = {0u, 0u};
    e = cudaMemcpyToSymbol(g_device_status, zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear device status");
    if (v[1] != 0) {
      // codes 0xB0000001..4: cu_seqlens; 0xB0000005 / 6: seqused_q / seqused_k
      const char* what = v[1] == 0xB0000005u   ? "seqused_q"
                         : v[1] == 0xB0000006u ? "seqused_k"
                                               : "cu_seqlens";
      return fail(ATTN_ERR_ARG, "%s failed device-side validation (code 0x%08x)", what, v[1]);
    }
    return fail(ATTN_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (site 0x%08x)", v[0]);
  }
  return ATTN_OK;
}

void attn_set_wait_timeout_ns(int64_t ns) {
  g_timeout_ns.store(ns > 0 ? static_cast<long long>(ns) : 4000000000LL);
}

const char* attn_last_error(void) { return g_err.c_str(); }

const char* attn_version(void) { return "attn_gb300 0.1.0 (sm_103a)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_bwd_noalloc: attn_bwd whose workspace is a fixed array in device memory
// owned by the library, for callers that may not allocate (include/attn_bwd.h
// says who and why).  The array is a file-scope __device__ variable, so every
// GPU that loads this library holds kNoAllocScratchBytes of it until the
// process exits.  In host code the name g_attn_noalloc_scratch is only a
// host-side handle; the kernels get the device address from
// cudaGetSymbolAddress, looked up once per device.

static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[32u << 20];

namespace {

constexpr size_t kNoAllocScratchBytes = sizeof(g_attn_noalloc_scratch);

// Device address of g_attn_noalloc_scratch on the current device.  The first
// call on a device does the lookup (with that device current) and caches it.
int noalloc_scratch(void** out) {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device index %d not supported", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch array");
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                                const attn_tensor* o, const float* lse, const attn_tensor* dout,
                                const attn_tensor* dq, const attn_tensor* dk,
                                const attn_tensor* dv, int dtype, int batch, int seqlen_q,
                                int seqlen_k, int h_q, int h_k, int head_dim, float scale,
                                int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
                                int max_seqlen_q, int max_seqlen_k, int deterministic,
                                attn_stream_t stream) {
  g_err.clear();
  int rc = check_common(dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, scale,
                        cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k);
  if (rc) return rc;
  const WsLayout w =
      ws_layout(batch, seqlen_q, h_q, head_dim, cu_seqlens_q != nullptr ? 1 : 0);
  if (w.total > kNoAllocScratchBytes)
    return fail(ATTN_ERR_WORKSPACE,
                "attn_bwd_noalloc: this problem needs %zu bytes of workspace but the library's "
                "static scratch holds %zu; use attn_bwd with a caller-provided workspace",
                w.total, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  // The preprocess kernel of every call clears the parts of the workspace that
  // must start at zero (dQ accumulator, semaphores, work counter); the rest is
  // written before it is read.
  void* workspace = scratch;
  const size_t workspace_bytes = kNoAllocScratchBytes;
  return bwd_entry(kPre | kMain | kPost, ATTN_BWD_ARGS_PASS, stream);
}
