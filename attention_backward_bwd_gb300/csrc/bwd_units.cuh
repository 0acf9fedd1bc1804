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

// Unit order (the scheduler hands units out in index order; the launch sets
// p.unit_seq_major and p.unit_per).  Key-tile major, (n, b, g) with g innermost:
// the CTAs running at once hold the first key tiles (the longest units under a
// causal mask) of every (sequence, kv head) group, ~10 CTAs per group on the
// bench workload (GQA, 16 groups), sharing each group's Q/dO tiles and dQ
// accumulator rows in L2.  Sequence major, (b, n, g): packed (varlen) batches,
// where key-tile major spread the running CTAs over every group of 16 sequences
// x 16 heads and moved 41 GB of DRAM per launch (84 % of the DRAM peak; 5.5 GB
// sequence major), and, in the D = 128 main kernel, padded MHA batches outside
// deterministic mode (~10 CTAs per head instead of ~5: MHA S = 4096 non-causal
// +3.4 %; GQA groups are shared enough already, and deterministic mode's longer
// chains and the other kernels lose by it).  Either way each group's key tiles
// come in ascending order: longest first, and the order the deterministic
// mode's semaphores expect.  The decode has no branch on the order: an earlier
// form that chose it by a branch on the sequence layout slowed the short-unit
// D = 64 kernel by 12 %.
// win_left: the left window side (-1 = none; a compile-time -1 in the
// instantiation without a left window), win_right: p.win_right.
__device__ __forceinline__ Unit get_unit(const BwdParams& p, int u, int G, int win_left) {
  Unit r;
  const int outer = u / p.unit_per;
  const int rem = u - outer * p.unit_per;
  const int mid = rem / p.h_k;
  r.g = rem - mid * p.h_k;
  r.n = p.unit_seq_major ? mid : outer;
  r.b = p.unit_seq_major ? outer : mid;
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
