// Work units of the KV-stationary backward kernels: one unit = (key tile n of
// 128 keys, key/value head g, sequence b), iterated over the query heads of
// the group and the query tiles that see key tile n.
#pragma once

#include "common.cuh"

namespace attn {

struct Unit {
  int n, g, b;
  SeqInfo si;
  int m_start, m_count, n_iters;
  bool has_keys;
};

// Unit order (the scheduler hands units out in index order): padded batches are
// key-tile major, (n, b, g) with g innermost, so the CTAs running at once are
// the first key tiles (the longest units under a causal mask) of every
// (sequence, kv head) group.  Packed varlen batches are sequence major, (b, n,
// g): with many sequences, key-tile major would spread the running CTAs over
// every group, and their Q/dO tiles and dQ accumulator rows would not stay in
// L2 (measured: 41 GB of DRAM traffic per launch for 16 sequences of up to 8192,
// 84 % of the DRAM peak); sequence major keeps them on one sequence's groups,
// each group's key tiles still in ascending order (longest first, and the order
// the deterministic mode's semaphores expect).  With seq_major_mha (the D = 128
// main kernel) padded MHA batches (one query head per group) outside
// deterministic mode take the sequence-major order too: it shares each head's
// tiles among ~10 running CTAs instead of ~5 (MHA S = 4096 non-causal +3.4 %);
// GQA groups are already shared enough, and the longer deterministic chains and
// the other kernels lose by it.
// win_left: the left window side (-1 = none; a compile-time -1 in the
// instantiation without a left window), win_right: p.win_right.
__device__ __forceinline__ Unit get_unit(const BwdParams& p, int u, int G, int win_left,
                                         bool seq_major_mha) {
  Unit r;
  if (p.seq.cu_q != nullptr || (seq_major_mha && G == 1 && !p.deterministic)) {
    const int per_b = (p.max_seqlen_k + kTileRows - 1) / kTileRows * p.h_k;
    r.b = u / per_b;
    const int rem = u - r.b * per_b;
    r.n = rem / p.h_k;
    r.g = rem - r.n * p.h_k;
  } else {
    const int per_n = p.seq.batch * p.h_k;
    r.n = u / per_n;
    const int rem = u - r.n * per_n;
    r.b = rem / p.h_k;
    r.g = rem - r.b * p.h_k;
  }
  r.si = seq_info(p.seq, r.b);
  r.has_keys = r.n * kTileRows < r.si.sk;
  // query tiles holding a query that sees a key of this tile (all of them
  // without a mask; causal or a window narrows the range)
  const int k1 = min(r.n * kTileRows + kTileRows, r.si.sk);
  int lo, hi;
  window_queries(r.n * kTileRows, k1, r.si.sq, r.si.sk, win_left, p.win_right, lo, hi);
  r.m_start = lo / kTileRows;
  r.m_count = lo < hi ? ceil_div(hi, kTileRows) - r.m_start : 0;
  r.n_iters = r.has_keys ? G * r.m_count : 0;
  return r;
}

// Iteration j of a unit -> (query head h, query tile m), heads of the group
// innermost.  Query tiles run from the last to the first, so every CTA working
// on the same (sequence, kv head) reads the same Q/dO tile at about the same
// time (the causal start tile only shortens the tail) and those tiles are
// served from L2 instead of being streamed from HBM once per key tile.  The
// same order serves deterministic mode: key tiles that start together meet
// each query tile together, so key tile n trails key tile n-1 only by the
// latency of one ordered add.  (First to last would put key tile n one query
// tile ahead of key tile n-1 from the start, a wait of G tiles per link of the
// chain; measured 10 % slower.)
__device__ __forceinline__ void iter_hm(const Unit& un, int j, int G, int& h, int& m) {
  const int jm = j / G;
  h = un.g * G + (j - jm * G);
  m = un.m_start + un.m_count - 1 - jm;
}

}  // namespace attn
