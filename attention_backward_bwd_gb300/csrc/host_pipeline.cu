// attn_bwd_host: the backward for tensors that live in host memory.
//
// The inputs go to the device, the three backward kernels run, and dQ, dK, dV
// come back, all inside one call.  Done in that order the copies and the
// kernels never overlap: at B=2, H_q=32, H_k=8, S=8192, D=128 the copies
// (472 MB in, 201 MB out) take longer than the kernels.  So the problem is cut
// into chunks that are independent backward problems (whole key/value head
// groups of one sequence, or whole sequences), and the chunks flow through
// three kinds of internal streams:
//   copy-in stream   H2D of chunk 0, 1, 2, ...        (one stream: the H2D engine is serial)
//   compute streams  preprocess/main/postprocess of chunk c on stream c % 3,
//                    after chunk c's copy-in event; chunk c's workspace is
//                    slot c % 3, free again once chunk c - 3 (same stream) is done
//   copy-out stream  D2H of chunk c after chunk c's compute event
// so chunk c+1 is copied in and chunk c-1 copied out while chunk c computes,
// and one chunk's kernels can fill the SMs that the previous chunk's kernels
// leave idle at their tail (a chunk's longest work unit can last longer than
// its share of the step, hence three compute streams rather than two).
// Measured on one GB300 at the workload above: H2D 204-210 GB/s, D2H 183-193
// GB/s, both at once 336 GB/s in total, so the copies in alone take ~2.3 ms
// against 2.63 ms of kernels; 8 chunks and 3 compute streams give 3.42 ms per
// call (2 streams: 3.73 ms; 16 chunks: 4.6 ms, 4 streams 3.7 ms).
// Every internal stream first waits for the caller's stream, and the caller's
// stream then waits for the copy-out stream, so the call is ordered like any
// other work on the caller's stream.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/attn_bwd.h"
#include "internal.h"

namespace attn {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;
constexpr int kSlots = 3;  // compute streams = workspaces

// Streams and events of one device, created on first use and kept for the
// life of the process.  An event may be re-recorded by a later call: a wait
// that was already enqueued keeps the state the event had at that time.
struct Pool {
  bool ready;
  cudaStream_t in, out, comp[kSlots];
  cudaEvent_t start, done, in_done[kMaxChunks], comp_done[kMaxChunks];
};

Pool g_pool[kMaxDevices];
std::mutex g_pool_mu;

void destroy_pool(Pool& t) {
  cudaStream_t streams[2 + kSlots] = {t.in, t.out};
  for (int i = 0; i < kSlots; ++i) streams[2 + i] = t.comp[i];
  for (cudaStream_t st : streams)
    if (st != nullptr) cudaStreamDestroy(st);
  cudaEvent_t single[2] = {t.start, t.done};
  for (cudaEvent_t ev : single)
    if (ev != nullptr) cudaEventDestroy(ev);
  for (int i = 0; i < kMaxChunks; ++i) {
    if (t.in_done[i] != nullptr) cudaEventDestroy(t.in_done[i]);
    if (t.comp_done[i] != nullptr) cudaEventDestroy(t.comp_done[i]);
  }
}

int get_pool(Pool** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(ATTN_ERR_CUDA, "device index %d not supported", dev);
  Pool& P = g_pool[dev];
  if (!P.ready) {
    // build into a zeroed pool; on a failure destroy what was made, so a later
    // call starts again from nothing
    Pool t = {};
    const unsigned sflags = cudaStreamNonBlocking;
    const unsigned eflags = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&t.in, sflags);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&t.out, sflags);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i)
      e = cudaStreamCreateWithFlags(&t.comp[i], sflags);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t.start, eflags);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t.done, eflags);
    for (int i = 0; i < kMaxChunks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&t.in_done[i], eflags);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t.comp_done[i], eflags);
    }
    if (e != cudaSuccess) {
      destroy_pool(t);
      return cuda_fail(e, "create the internal streams and events");
    }
    t.ready = true;
    P = t;
  }
  *out = &P;
  return ATTN_OK;
}

// How the problem is cut.  With batch >= want, each chunk is a run of
// `seqs` whole sequences (all heads); otherwise each chunk is one sequence
// and `kv_heads` consecutive key/value heads (with their query-head groups),
// kv_heads the largest divisor of h_k that still gives at least `want` chunks
// (or 1).
struct Chunking {
  int seqs, kv_heads, n;
};

Chunking chunking(int batch, int h_k, int want) {
  if (want <= 0) want = 8;
  if (want > kMaxChunks) want = kMaxChunks;
  Chunking c;
  if (batch >= want) {
    c.seqs = (batch + want - 1) / want;
    c.kv_heads = h_k;
    c.n = (batch + c.seqs - 1) / c.seqs;
    return c;
  }
  c.seqs = 1;
  c.kv_heads = 1;
  for (int d = h_k; d >= 1; --d)
    if (h_k % d == 0 && static_cast<int64_t>(batch) * (h_k / d) >= want) {
      c.kv_heads = d;
      break;
    }
  c.n = batch * (h_k / c.kv_heads);
  if (c.n > kMaxChunks) {  // only if h_k has no divisor in between: fall back to whole heads
    c.kv_heads = h_k;
    c.n = batch;
  }
  return c;
}

// Device buffer: compact [B, S, H, D] copies of the eight tensors, LSE
// [B, H_q, Sq], then one workspace per compute stream sized for a chunk.
struct BufLayout {
  size_t q, k, v, o, dout, dq, dk, dv, lse, ws[kSlots], ws_bytes, total;
};

BufLayout buf_layout(int batch, int seqlen_q, int seqlen_k, int h_q, int h_k, int head_dim,
                     const Chunking& c) {
  const size_t e = 2;
  const size_t nq = static_cast<size_t>(batch) * seqlen_q * h_q * head_dim * e;
  const size_t nk = static_cast<size_t>(batch) * seqlen_k * h_k * head_dim * e;
  BufLayout L;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t off = at;
    at = align256(at + bytes);
    return off;
  };
  L.q = take(nq);
  L.o = take(nq);
  L.dout = take(nq);
  L.dq = take(nq);
  L.k = take(nk);
  L.v = take(nk);
  L.dk = take(nk);
  L.dv = take(nk);
  L.lse = take(static_cast<size_t>(batch) * h_q * seqlen_q * 4);
  const int g = h_q / h_k;
  L.ws_bytes = ws_layout(c.seqs, seqlen_q, c.kv_heads * g, head_dim, 0).total;
  for (int i = 0; i < kSlots; ++i) L.ws[i] = take(L.ws_bytes);
  L.total = at;
  return L;
}

int check_host_tensor(const attn_tensor* t, const char* name, int heads, int head_dim, int rows,
                      bool need) {
  if (t == nullptr) return fail(ATTN_ERR_NULL, "%s: descriptor is NULL", name);
  if (!need) return ATTN_OK;
  if (t->ptr == nullptr) return fail(ATTN_ERR_NULL, "%s: pointer is NULL", name);
  if (t->stride_h != head_dim)
    return fail(ATTN_ERR_STRIDE,
                "%s: host tensors need adjacent heads (stride_h == D = %d, got %lld)", name,
                head_dim, static_cast<long long>(t->stride_h));
  if (t->stride_s < static_cast<int64_t>(heads) * head_dim ||
      t->stride_b < static_cast<int64_t>(rows) * t->stride_s)
    return fail(ATTN_ERR_STRIDE, "%s: strides overlap (s=%lld, b=%lld)", name,
                static_cast<long long>(t->stride_s), static_cast<long long>(t->stride_b));
  return ATTN_OK;
}

attn_tensor compact_view(char* base, int seqlen, int heads, int head_dim) {
  const int64_t ss = static_cast<int64_t>(heads) * head_dim;
  return attn_tensor{base, ss * seqlen, ss, head_dim};
}

// Copies rows [0, seqlen) of heads [h0, h0 + nh) of sequences [b0, b0 + nb)
// between a host tensor and the compact device copy (to_device selects the
// direction), one 2-D copy per sequence.
cudaError_t copy_heads(const attn_tensor& host, char* dev, int b0, int nb, int h0, int nh,
                       int seqlen, int heads, int head_dim, bool to_device, cudaStream_t st) {
  if (seqlen == 0 || nh == 0) return cudaSuccess;
  const size_t e = 2;
  const size_t width = static_cast<size_t>(nh) * head_dim * e;
  const size_t dpitch = static_cast<size_t>(heads) * head_dim * e;
  for (int b = b0; b < b0 + nb; ++b) {
    char* h = static_cast<char*>(host.ptr) +
              (static_cast<int64_t>(b) * host.stride_b + static_cast<int64_t>(h0) * head_dim) * e;
    char* d = dev + ((static_cast<size_t>(b) * seqlen) * heads + h0) * head_dim * e;
    const size_t hpitch = static_cast<size_t>(host.stride_s) * e;
    const cudaError_t r =
        to_device ? cudaMemcpy2DAsync(d, dpitch, h, hpitch, width, seqlen, cudaMemcpyDefault, st)
                  : cudaMemcpy2DAsync(h, hpitch, d, dpitch, width, seqlen, cudaMemcpyDefault, st);
    if (r != cudaSuccess) return r;
  }
  return cudaSuccess;
}

// The stream and event choreography shared by both entry points: every
// internal stream waits for the caller's stream; `prologue` runs first on the
// copy-in stream; chunk c's copies in run on the copy-in stream, its kernels on
// compute stream c % kSlots (workspace slot c % kSlots) after them, and its
// copies out on the copy-out stream after the kernels; the caller's stream
// then waits for the copy-out stream.  Each callback returns ATTN_OK or an
// error code (with the message already set).
template <typename Prologue, typename CopyIn, typename Compute, typename CopyOut>
int run_chunks(cudaStream_t user, int n, Prologue prologue, CopyIn copy_in, Compute compute,
               CopyOut copy_out) {
  std::lock_guard<std::mutex> lock(g_pool_mu);
  Pool* P = nullptr;
  int rc = get_pool(&P);
  if (rc) return rc;
  cudaError_t e;
  if ((e = cudaEventRecord(P->start, user)) != cudaSuccess) return cuda_fail(e, "record start");
  cudaStream_t all[2 + kSlots];
  all[0] = P->in;
  all[1] = P->out;
  for (int i = 0; i < kSlots; ++i) all[2 + i] = P->comp[i];
  for (cudaStream_t s : all)
    if ((e = cudaStreamWaitEvent(s, P->start, 0)) != cudaSuccess) return cuda_fail(e, "wait start");
  if ((rc = prologue(P->in))) return rc;
  for (int c = 0; c < n; ++c) {
    if ((rc = copy_in(c, P->in))) return rc;
    if ((e = cudaEventRecord(P->in_done[c], P->in)) != cudaSuccess) return cuda_fail(e, "record");
    cudaStream_t cs = P->comp[c % kSlots];
    if ((e = cudaStreamWaitEvent(cs, P->in_done[c], 0)) != cudaSuccess)
      return cuda_fail(e, "wait copy-in");
    if ((rc = compute(c, c % kSlots, cs))) return rc;
    if ((e = cudaEventRecord(P->comp_done[c], cs)) != cudaSuccess) return cuda_fail(e, "record");
    if ((e = cudaStreamWaitEvent(P->out, P->comp_done[c], 0)) != cudaSuccess)
      return cuda_fail(e, "wait compute");
    if ((rc = copy_out(c, P->out))) return rc;
  }
  if ((e = cudaEventRecord(P->done, P->out)) != cudaSuccess) return cuda_fail(e, "record done");
  if ((e = cudaStreamWaitEvent(user, P->done, 0)) != cudaSuccess) return cuda_fail(e, "wait done");
  return ATTN_OK;
}

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" size_t attn_bwd_host_buffer_size(int batch, int seqlen_q, int seqlen_k, int h_q,
                                            int h_k, int head_dim, int chunks) {
  if (batch <= 0 || seqlen_q < 0 || seqlen_k < 0 || h_q <= 0 || h_k <= 0 || h_q % h_k != 0 ||
      head_dim <= 0)
    return 0;
  return buf_layout(batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, chunking(batch, h_k, chunks))
      .total;
}

extern "C" int attn_bwd_host(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                             const attn_tensor* o, const float* lse, const attn_tensor* dout,
                             const attn_tensor* dq, const attn_tensor* dk, const attn_tensor* dv,
                             int dtype, int batch, int seqlen_q, int seqlen_k, int h_q, int h_k,
                             int head_dim, float scale, int causal, int deterministic,
                             const attn_opts* opts, int chunks, void* device_buffer,
                             size_t device_buffer_bytes, attn_stream_t stream) {
  clear_error();
  int rc = check_common(dtype, batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, scale, nullptr,
                        nullptr, 0, 0);
  if (rc) return rc;
  const bool hq = seqlen_q > 0, hk = seqlen_k > 0;
  if ((rc = check_host_tensor(q, "q", h_q, head_dim, seqlen_q, hq && hk))) return rc;
  if ((rc = check_host_tensor(k, "k", h_k, head_dim, seqlen_k, hq && hk))) return rc;
  if ((rc = check_host_tensor(v, "v", h_k, head_dim, seqlen_k, hq && hk))) return rc;
  if ((rc = check_host_tensor(o, "o", h_q, head_dim, seqlen_q, hq && hk))) return rc;
  if ((rc = check_host_tensor(dout, "dout", h_q, head_dim, seqlen_q, hq && hk))) return rc;
  if ((rc = check_host_tensor(dq, "dq", h_q, head_dim, seqlen_q, hq))) return rc;
  if ((rc = check_host_tensor(dk, "dk", h_k, head_dim, seqlen_k, hk))) return rc;
  if ((rc = check_host_tensor(dv, "dv", h_k, head_dim, seqlen_k, hk))) return rc;
  if (hq && hk && lse == nullptr) return fail(ATTN_ERR_NULL, "lse is NULL");
  attn_opts checked;
  if ((rc = resolve_opts(opts, &checked))) return rc;
  if (checked.seqused_q != nullptr || checked.seqused_k != nullptr)
    return fail(ATTN_ERR_ARG, "seqused_q/k are not taken by the host-buffer calls");
  const Chunking ch = chunking(batch, h_k, chunks);
  const BufLayout L = buf_layout(batch, seqlen_q, seqlen_k, h_q, h_k, head_dim, ch);
  if (device_buffer == nullptr) return fail(ATTN_ERR_WORKSPACE, "device_buffer is NULL");
  if (reinterpret_cast<uintptr_t>(device_buffer) % 256 != 0)
    return fail(ATTN_ERR_WORKSPACE, "device_buffer must be 256-byte aligned");
  if (device_buffer_bytes < L.total)
    return fail(ATTN_ERR_WORKSPACE, "device_buffer too small: %zu bytes given, %zu needed",
                device_buffer_bytes, L.total);

  char* buf = static_cast<char*>(device_buffer);
  const int g = h_q / h_k;
  // chunk c: sequences [b0, b0 + nb), kv heads [j0, j0 + nj), query heads [i0, i0 + ni)
  auto geom = [&](int c, int& b0, int& nb, int& j0, int& nj, int& i0, int& ni) {
    b0 = (ch.kv_heads == h_k) ? c * ch.seqs : c / (h_k / ch.kv_heads);
    nb = (ch.kv_heads == h_k) ? (b0 + ch.seqs <= batch ? ch.seqs : batch - b0) : 1;
    j0 = (ch.kv_heads == h_k) ? 0 : (c % (h_k / ch.kv_heads)) * ch.kv_heads;
    nj = ch.kv_heads;
    i0 = j0 * g;
    ni = nj * g;
  };
  auto copy_in = [&](int c, cudaStream_t st) -> int {
    if (!(hq && hk)) return ATTN_OK;
    int b0, nb, j0, nj, i0, ni;
    geom(c, b0, nb, j0, nj, i0, ni);
    cudaError_t e;
    // Q, O, dO, K, V slices and the chunk's LSE rows (contiguous in [B, H_q, Sq])
    if ((e = copy_heads(*q, buf + L.q, b0, nb, i0, ni, seqlen_q, h_q, head_dim, true, st)) ||
        (e = copy_heads(*o, buf + L.o, b0, nb, i0, ni, seqlen_q, h_q, head_dim, true, st)) ||
        (e = copy_heads(*dout, buf + L.dout, b0, nb, i0, ni, seqlen_q, h_q, head_dim, true, st)) ||
        (e = copy_heads(*k, buf + L.k, b0, nb, j0, nj, seqlen_k, h_k, head_dim, true, st)) ||
        (e = copy_heads(*v, buf + L.v, b0, nb, j0, nj, seqlen_k, h_k, head_dim, true, st)))
      return cuda_fail(e, "copy inputs to the device");
    const size_t lse_off = (static_cast<size_t>(b0) * h_q + i0) * seqlen_q;
    const size_t lse_n = static_cast<size_t>(nb) * ni * seqlen_q;
    if ((e = cudaMemcpyAsync(buf + L.lse + lse_off * 4, lse + lse_off, lse_n * 4,
                             cudaMemcpyDefault, st)) != cudaSuccess)
      return cuda_fail(e, "copy lse to the device");
    return ATTN_OK;
  };
  auto compute = [&](int c, int slot, cudaStream_t cs) -> int {
    // the chunk is a backward problem of nb sequences and ni / nj heads
    int b0, nb, j0, nj, i0, ni;
    geom(c, b0, nb, j0, nj, i0, ni);
    const size_t qoff = (static_cast<size_t>(b0) * seqlen_q * h_q + i0) * head_dim * 2;
    const size_t koff = (static_cast<size_t>(b0) * seqlen_k * h_k + j0) * head_dim * 2;
    const attn_tensor tq = compact_view(buf + L.q + qoff, seqlen_q, h_q, head_dim);
    const attn_tensor to = compact_view(buf + L.o + qoff, seqlen_q, h_q, head_dim);
    const attn_tensor tdo = compact_view(buf + L.dout + qoff, seqlen_q, h_q, head_dim);
    const attn_tensor tdq = compact_view(buf + L.dq + qoff, seqlen_q, h_q, head_dim);
    const attn_tensor tk = compact_view(buf + L.k + koff, seqlen_k, h_k, head_dim);
    const attn_tensor tv = compact_view(buf + L.v + koff, seqlen_k, h_k, head_dim);
    const attn_tensor tdk = compact_view(buf + L.dk + koff, seqlen_k, h_k, head_dim);
    const attn_tensor tdv = compact_view(buf + L.dv + koff, seqlen_k, h_k, head_dim);
    const float* tlse = reinterpret_cast<const float*>(buf + L.lse) +
                        (static_cast<size_t>(b0) * h_q + i0) * seqlen_q;
    Prepared pr;
    int r = prepare_bwd(&tq, &tk, &tv, &to, tlse, &tdo, &tdq, &tdk, &tdv, dtype, nb, seqlen_q,
                        seqlen_k, ni, nj, head_dim, scale, causal, nullptr, nullptr, seqlen_q,
                        seqlen_k, deterministic, &checked, buf + L.ws[slot], L.ws_bytes, &pr);
    return r ? r : run_stages(kPre | kMain | kPost, pr, cs);
  };
  auto copy_out = [&](int c, cudaStream_t st) -> int {
    int b0, nb, j0, nj, i0, ni;
    geom(c, b0, nb, j0, nj, i0, ni);
    cudaError_t e;
    if ((e = copy_heads(*dq, buf + L.dq, b0, nb, i0, ni, seqlen_q, h_q, head_dim, false, st)) ||
        (e = copy_heads(*dk, buf + L.dk, b0, nb, j0, nj, seqlen_k, h_k, head_dim, false, st)) ||
        (e = copy_heads(*dv, buf + L.dv, b0, nb, j0, nj, seqlen_k, h_k, head_dim, false, st)))
      return cuda_fail(e, "copy results to the host");
    return ATTN_OK;
  };
  return run_chunks(reinterpret_cast<cudaStream_t>(stream), ch.n,
                    [](cudaStream_t) { return static_cast<int>(ATTN_OK); }, copy_in, compute,
                    copy_out);
}

// ---------------------------------------------------------------------------
// attn_bwd_host_varlen: the same pipeline for packed [total, H, D] tensors.
// A chunk is a run of whole sequences (all heads), the runs cut so that each
// holds about an equal share of the attention work (query rows x key rows per
// sequence); its rows are contiguous, so each tensor moves in one pitched copy.
// The chunk's LSE rows, which are strided in [H_q, total_q], land in a compact
// [H_q, rows] block of their own, and its cu_seqlens are rebased to start at 0
// (all chunks' arrays go to the device in one small copy before the first).

namespace attn {
namespace {

struct VarlenChunk {
  int b0, nb;          // sequences [b0, b0 + nb)
  int q0, nq, k0, nk;  // packed rows [q0, q0 + nq) and [k0, k0 + nk)
  int max_q, max_k;    // longest query / key sequence of the chunk
  int cu_off;          // offset (in ints) of the chunk's rebased cu_q; cu_k follows
};

int plan_varlen(const int* cu_q, const int* cu_k, int batch, int total_q, int total_k, int want,
                VarlenChunk* out, int* n_out) {
  if (cu_q == nullptr || cu_k == nullptr) return fail(ATTN_ERR_NULL, "cu_seqlens is NULL");
  if (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[batch] != total_q || cu_k[batch] != total_k)
    return fail(ATTN_ERR_ARG, "cu_seqlens must start at 0 and end at the total row counts");
  double work = 0;
  for (int b = 0; b < batch; ++b) {
    const int lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
    if (lq < 0 || lk < 0) return fail(ATTN_ERR_ARG, "cu_seqlens must be nondecreasing");
    work += static_cast<double>(lq) * lk + lq + lk;
  }
  if (want <= 0) want = 8;
  if (want > kMaxChunks) want = kMaxChunks;
  const double share = work / want;
  int n = 0, b = 0, cu_off = 0;
  while (b < batch) {
    VarlenChunk c{b, 0, cu_q[b], 0, cu_k[b], 0, 0, 0, cu_off};
    double w = 0;
    // take sequences until the share is reached; the last chunk takes the rest
    while (b < batch && (c.nb == 0 || w < share || n == want - 1)) {
      const int lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
      w += static_cast<double>(lq) * lk + lq + lk;
      c.max_q = lq > c.max_q ? lq : c.max_q;
      c.max_k = lk > c.max_k ? lk : c.max_k;
      ++c.nb;
      ++b;
    }
    c.nq = cu_q[b] - c.q0;
    c.nk = cu_k[b] - c.k0;
    cu_off += 2 * (c.nb + 1);
    out[n++] = c;
  }
  *n_out = n;
  return ATTN_OK;
}

struct VarlenLayout {
  size_t q, k, v, o, dout, dq, dk, dv, lse, cu, ws[kSlots], ws_bytes, total;
};

VarlenLayout varlen_layout(int batch, int total_q, int total_k, int h_q, int h_k, int head_dim,
                           const VarlenChunk* ch, int n) {
  const size_t e = 2;
  const size_t nq = static_cast<size_t>(total_q) * h_q * head_dim * e;
  const size_t nk = static_cast<size_t>(total_k) * h_k * head_dim * e;
  VarlenLayout L;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t off = at;
    at = align256(at + bytes);
    return off;
  };
  L.q = take(nq);
  L.o = take(nq);
  L.dout = take(nq);
  L.dq = take(nq);
  L.k = take(nk);
  L.v = take(nk);
  L.dk = take(nk);
  L.dv = take(nk);
  L.lse = take(static_cast<size_t>(h_q) * total_q * 4);
  L.cu = take(static_cast<size_t>(2) * (batch + n) * 4);
  L.ws_bytes = 0;
  for (int c = 0; c < n; ++c) {
    const size_t w = ws_layout(ch[c].nb, ch[c].nq, h_q, head_dim, 1).total;
    L.ws_bytes = w > L.ws_bytes ? w : L.ws_bytes;
  }
  for (int i = 0; i < kSlots; ++i) L.ws[i] = take(L.ws_bytes);
  L.total = at;
  return L;
}

// rows [r0, r0 + n) of a packed host tensor <-> the same rows of its compact
// device copy, all heads, one pitched copy
cudaError_t copy_rows(const attn_tensor& host, char* dev, int r0, int n, int heads, int head_dim,
                      bool to_device, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const size_t e = 2;
  const size_t width = static_cast<size_t>(heads) * head_dim * e;
  const size_t hpitch = static_cast<size_t>(host.stride_s) * e;
  char* h = static_cast<char*>(host.ptr) + static_cast<int64_t>(r0) * host.stride_s * e;
  char* d = dev + static_cast<size_t>(r0) * width;
  return to_device ? cudaMemcpy2DAsync(d, width, h, hpitch, width, n, cudaMemcpyDefault, st)
                   : cudaMemcpy2DAsync(h, hpitch, d, width, width, n, cudaMemcpyDefault, st);
}

int check_packed_host_tensor(const attn_tensor* t, const char* name, int heads, int head_dim,
                             bool need) {
  if (t == nullptr) return fail(ATTN_ERR_NULL, "%s: descriptor is NULL", name);
  if (!need) return ATTN_OK;
  if (t->ptr == nullptr) return fail(ATTN_ERR_NULL, "%s: pointer is NULL", name);
  if (t->stride_h != head_dim)
    return fail(ATTN_ERR_STRIDE,
                "%s: host tensors need adjacent heads (stride_h == D = %d, got %lld)", name,
                head_dim, static_cast<long long>(t->stride_h));
  if (t->stride_s < static_cast<int64_t>(heads) * head_dim)
    return fail(ATTN_ERR_STRIDE, "%s: rows overlap (stride_s=%lld)", name,
                static_cast<long long>(t->stride_s));
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" size_t attn_bwd_host_varlen_buffer_size(const int* cu_seqlens_q,
                                                   const int* cu_seqlens_k, int batch,
                                                   int total_q, int total_k, int h_q, int h_k,
                                                   int head_dim, int chunks) {
  if (batch <= 0 || total_q < 0 || total_k < 0 || h_q <= 0 || h_k <= 0 || h_q % h_k != 0 ||
      head_dim <= 0)
    return 0;
  VarlenChunk ch[kMaxChunks];
  int n = 0;
  if (plan_varlen(cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, chunks, ch, &n))
    return 0;  // invalid cu_seqlens (the message stays in attn_last_error)
  return varlen_layout(batch, total_q, total_k, h_q, h_k, head_dim, ch, n).total;
}

extern "C" int attn_bwd_host_varlen(const attn_tensor* q, const attn_tensor* k,
                                    const attn_tensor* v, const attn_tensor* o, const float* lse,
                                    const attn_tensor* dout, const attn_tensor* dq,
                                    const attn_tensor* dk, const attn_tensor* dv, int dtype,
                                    int batch, int total_q, int total_k, int h_q, int h_k,
                                    int head_dim, float scale, int causal,
                                    const int* cu_seqlens_q, const int* cu_seqlens_k,
                                    int deterministic, const attn_opts* opts, int chunks,
                                    void* device_buffer, size_t device_buffer_bytes,
                                    attn_stream_t stream) {
  clear_error();
  int rc = check_common(dtype, batch, total_q, total_k, h_q, h_k, head_dim, scale, nullptr,
                        nullptr, 0, 0);
  if (rc) return rc;
  const bool hq = total_q > 0, hk = total_k > 0;
  if ((rc = check_packed_host_tensor(q, "q", h_q, head_dim, hq && hk))) return rc;
  if ((rc = check_packed_host_tensor(k, "k", h_k, head_dim, hq && hk))) return rc;
  if ((rc = check_packed_host_tensor(v, "v", h_k, head_dim, hq && hk))) return rc;
  if ((rc = check_packed_host_tensor(o, "o", h_q, head_dim, hq && hk))) return rc;
  if ((rc = check_packed_host_tensor(dout, "dout", h_q, head_dim, hq && hk))) return rc;
  if ((rc = check_packed_host_tensor(dq, "dq", h_q, head_dim, hq))) return rc;
  if ((rc = check_packed_host_tensor(dk, "dk", h_k, head_dim, hk))) return rc;
  if ((rc = check_packed_host_tensor(dv, "dv", h_k, head_dim, hk))) return rc;
  if (hq && hk && lse == nullptr) return fail(ATTN_ERR_NULL, "lse is NULL");
  attn_opts checked;
  if ((rc = resolve_opts(opts, &checked))) return rc;
  if (checked.seqused_q != nullptr || checked.seqused_k != nullptr)
    return fail(ATTN_ERR_ARG, "seqused_q/k are not taken by the host-buffer calls");
  VarlenChunk ch[kMaxChunks];
  int n = 0;
  if ((rc = plan_varlen(cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, chunks, ch, &n)))
    return rc;
  const VarlenLayout L = varlen_layout(batch, total_q, total_k, h_q, h_k, head_dim, ch, n);
  if (device_buffer == nullptr) return fail(ATTN_ERR_WORKSPACE, "device_buffer is NULL");
  if (reinterpret_cast<uintptr_t>(device_buffer) % 256 != 0)
    return fail(ATTN_ERR_WORKSPACE, "device_buffer must be 256-byte aligned");
  if (device_buffer_bytes < L.total)
    return fail(ATTN_ERR_WORKSPACE, "device_buffer too small: %zu bytes given, %zu needed",
                device_buffer_bytes, L.total);
  // every chunk's rebased cu_seqlens_q then cu_seqlens_k
  std::vector<int> cu_all(static_cast<size_t>(2) * (batch + n));
  for (int c = 0; c < n; ++c) {
    int* dst = cu_all.data() + ch[c].cu_off;
    for (int i = 0; i <= ch[c].nb; ++i) {
      dst[i] = cu_seqlens_q[ch[c].b0 + i] - ch[c].q0;
      dst[ch[c].nb + 1 + i] = cu_seqlens_k[ch[c].b0 + i] - ch[c].k0;
    }
  }

  char* buf = static_cast<char*>(device_buffer);
  auto prologue = [&](cudaStream_t st) -> int {
    // pageable source: the call returns once the data sit in the driver's staging memory
    const cudaError_t e = cudaMemcpyAsync(buf + L.cu, cu_all.data(), cu_all.size() * sizeof(int),
                                          cudaMemcpyHostToDevice, st);
    return e == cudaSuccess ? static_cast<int>(ATTN_OK)
                            : cuda_fail(e, "copy cu_seqlens to the device");
  };
  auto lse_dev = [&](const VarlenChunk& C) {
    return reinterpret_cast<float*>(buf + L.lse) + static_cast<size_t>(h_q) * C.q0;
  };
  auto copy_in = [&](int c, cudaStream_t st) -> int {
    const VarlenChunk& C = ch[c];
    if (!(hq && hk)) return ATTN_OK;
    cudaError_t e;
    if ((e = copy_rows(*q, buf + L.q, C.q0, C.nq, h_q, head_dim, true, st)) ||
        (e = copy_rows(*o, buf + L.o, C.q0, C.nq, h_q, head_dim, true, st)) ||
        (e = copy_rows(*dout, buf + L.dout, C.q0, C.nq, h_q, head_dim, true, st)) ||
        (e = copy_rows(*k, buf + L.k, C.k0, C.nk, h_k, head_dim, true, st)) ||
        (e = copy_rows(*v, buf + L.v, C.k0, C.nk, h_k, head_dim, true, st)))
      return cuda_fail(e, "copy inputs to the device");
    // LSE [H_q, total_q]: the chunk's columns of every head, into a compact [H_q, nq]
    if (C.nq > 0 &&
        (e = cudaMemcpy2DAsync(lse_dev(C), static_cast<size_t>(C.nq) * 4, lse + C.q0,
                               static_cast<size_t>(total_q) * 4, static_cast<size_t>(C.nq) * 4,
                               h_q, cudaMemcpyDefault, st)) != cudaSuccess)
      return cuda_fail(e, "copy lse to the device");
    return ATTN_OK;
  };
  auto compute = [&](int c, int slot, cudaStream_t cs) -> int {
    const VarlenChunk& C = ch[c];
    const size_t qoff = static_cast<size_t>(C.q0) * h_q * head_dim * 2;
    const size_t koff = static_cast<size_t>(C.k0) * h_k * head_dim * 2;
    const int64_t sq = static_cast<int64_t>(h_q) * head_dim;
    const int64_t sk = static_cast<int64_t>(h_k) * head_dim;
    const attn_tensor tq{buf + L.q + qoff, 0, sq, head_dim}, to{buf + L.o + qoff, 0, sq, head_dim};
    const attn_tensor tdo{buf + L.dout + qoff, 0, sq, head_dim};
    const attn_tensor tdq{buf + L.dq + qoff, 0, sq, head_dim};
    const attn_tensor tk{buf + L.k + koff, 0, sk, head_dim}, tv{buf + L.v + koff, 0, sk, head_dim};
    const attn_tensor tdk{buf + L.dk + koff, 0, sk, head_dim};
    const attn_tensor tdv{buf + L.dv + koff, 0, sk, head_dim};
    const int* cuq = reinterpret_cast<const int*>(buf + L.cu) + C.cu_off;
    const int* cuk = cuq + C.nb + 1;
    Prepared pr;
    int r = prepare_bwd(&tq, &tk, &tv, &to, lse_dev(C), &tdo, &tdq, &tdk, &tdv, dtype, C.nb, C.nq,
                        C.nk, h_q, h_k, head_dim, scale, causal, cuq, cuk, C.max_q, C.max_k,
                        deterministic, &checked, buf + L.ws[slot], L.ws_bytes, &pr);
    return r ? r : run_stages(kPre | kMain | kPost, pr, cs);
  };
  auto copy_out = [&](int c, cudaStream_t st) -> int {
    const VarlenChunk& C = ch[c];
    cudaError_t e;
    if ((e = copy_rows(*dq, buf + L.dq, C.q0, C.nq, h_q, head_dim, false, st)) ||
        (e = copy_rows(*dk, buf + L.dk, C.k0, C.nk, h_k, head_dim, false, st)) ||
        (e = copy_rows(*dv, buf + L.dv, C.k0, C.nk, h_k, head_dim, false, st)))
      return cuda_fail(e, "copy results to the host");
    return ATTN_OK;
  };
  return run_chunks(reinterpret_cast<cudaStream_t>(stream), n, prologue, copy_in, compute,
                    copy_out);
}
