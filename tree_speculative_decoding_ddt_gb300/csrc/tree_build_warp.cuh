// A. Best-first draft-tree construction by one warp (device functions shared
// by the standalone tree-build kernel and the verify-attention kernel, which
// builds the tree in a spare warp while the prefix part of the attention
// runs).
//
// "The Milestone Commit: Cementing a Native DDTree Inference Engine",
// sections "What the Message Actually Does" and "The Reasoning Behind the
// Architecture": the builder replaces a CPU heapq, accumulates log-weights in
// double so that its pop order is bit-identical to the reference, keeps each
// node's ancestor set as a bitmask (parent mask | own bit) and emits the
// first-child / next-sibling encoding alongside tokens, parents and depths.
//
// The pop loop is a serial chain of at most budget steps, so only what the
// next pop depends on stays inside it: the frontier (at most budget+1 live
// entries, four per lane, in registers), a 32-lane argmax done with three
// redux.sync reductions on integer keys, and the two pushes. Node records
// (score and the popped entry's tie word) stay in the registers of lane
// n % 32; tokens, parents, depths, child lists and ancestor masks are derived
// from them after the loop.
//
// A frontier entry's tie word is depth | rank | parent | previous sibling,
// 8 bits each from the top. The first three order equal scores (lower depth,
// then lower rank, then lower parent index pops first) and identify the
// entry; the low byte records which popped node pushed a sibling entry, which
// gives the next-sibling links without any search. Pushes that can never be
// popped within the budget (depth or rank >= budget) are skipped: a node of
// depth d and rank r is popped at slot >= d + r.
#pragma once

#include <math.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace tb {

constexpr uint32_t kInvalid = 0xFFFFFFFFu;
constexpr uint32_t kNoPrev = 0xFFu;
constexpr int kSlots = kMaxQ / 32;  // most frontier entries and node records per lane
static_assert(kSlots == 4, "node records are four named registers per lane");

// Frontier slots per lane for Q tree slots: a frontier never holds more than
// Q entries (each pop removes one and adds at most two).
__host__ __device__ constexpr int slots_for(int Q) { return (Q + 31) / 32; }

// Tie words of the nodes lane, lane + 32, lane + 64, lane + 96 as popped:
// named registers, not an array, so that a record picked by a run-time slot
// index stays in registers (a select chain) instead of going to local memory.
struct NodeRecs {
  uint32_t t0 = 0u, t1 = 0u, t2 = 0u, t3 = 0u;
  __device__ __forceinline__ uint32_t tie(int k) const {
    return k == 0 ? t0 : k == 1 ? t1 : k == 2 ? t2 : t3;
  }
  __device__ __forceinline__ void set(int k, uint32_t t) {
    t0 = k == 0 ? t : t0;
    t1 = k == 1 ? t : t1;
    t2 = k == 2 ? t : t2;
    t3 = k == 3 ? t : t3;
  }
};

// Per-warp shared memory of one build (the staged candidate table follows it:
// log-probs as double, then token ids).
struct Smem {
  double score[kMaxQ];  // node scores (written by the pop loop)
  int32_t par[kMaxQ];
  int32_t dep[kMaxQ];
  int32_t tok[kMaxQ];
  int32_t fc[kMaxQ];
  int32_t ns[kMaxQ];
  unsigned long long anc[kMaxQ][kMaxW];
};

__host__ __device__ constexpr size_t smem_bytes(int De, int Ke) {
  return sizeof(Smem) + (size_t)De * Ke * (sizeof(double) + sizeof(int32_t));
}

// Order-preserving map of a double to a uint64: a larger score gives a larger
// key, -0.0 and +0.0 give the same key (they compare equal as doubles).
// GB300's FP64 pipe is narrow, so all comparisons run on these integer keys;
// only the two score additions per pop stay in FP64 (they must round exactly
// like the reference's double additions).
__device__ __forceinline__ unsigned long long score_key(double s) {
  unsigned long long u = (unsigned long long)__double_as_longlong(s);
  if (u == 0x8000000000000000ull) u = 0ull;
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_score(unsigned long long k) {
  const unsigned long long u = (k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
  return __longlong_as_double((long long)u);
}
__device__ __forceinline__ uint32_t tie_of(int d, int r, int par, uint32_t prev) {
  return ((uint32_t)d << 24) | ((uint32_t)r << 16) | ((uint32_t)par << 8) | prev;
}
// pop order: larger key first, then the smaller tie word
__device__ __forceinline__ bool before(unsigned long long ka, uint32_t ta, unsigned long long kb,
                                       uint32_t tb) {
  if (ta == kInvalid) return false;
  if (tb == kInvalid) return true;
  return ka > kb || (ka == kb && ta < tb);
}

// Builds the tree of one sequence with the calling warp (all 32 lanes).
// lp/ip: that sequence's [D][K] log-probs and token ids. De = min(D, budget),
// Ke = min(K, budget). On return S holds parents, depths, tokens, child links
// and ancestor words for every slot c < budget + 1 (slots past the tree: no
// parent, depth -1, token 0, own bit only). Returns the node count (1, the
// root alone, when the input is invalid; *bad then true).
template <int NS>  // frontier slots per lane: slots_for(budget + 1)
__device__ __forceinline__ int build_warp(const float* __restrict__ lp,
                                          const int32_t* __restrict__ ip, int32_t root, int D,
                                          int K, int budget, int V, int De, int Ke, Smem& S,
                                          double* s_logp, int32_t* s_ids, bool* bad_out) {
  const int lane = threadIdx.x & 31;
  const int Q = budget + 1;

  // ---- input validation over all D*K candidates ----------------------------
  bool bad = false;
  for (int e = lane; e < D * K; e += 32) {
    const float x = lp[e];
    const int32_t t = ip[e];
    bad |= !isfinite(x) || t < 0 || t >= V;
  }
  bad |= (root < 0 || root >= V);
  bad = __any_sync(0xffffffffu, bad);

  // ---- stage the reachable part of the candidate table ---------------------
  for (int e = lane; e < De * Ke; e += 32) {
    const int d = e / Ke, r = e % Ke;
    s_logp[e] = (double)lp[d * K + r];  // exact; done once, off the pop chain
    s_ids[e] = ip[d * K + r];
  }
  for (int c = lane; c < kMaxQ; c += 32) {
    S.fc[c] = -1;
    S.ns[c] = -1;
  }
  if (lane == 0) S.score[0] = 0.0;
  __syncwarp();

  // ---- frontier: position p lives in lane p % 32, slot p / 32 ---------------
  static_assert(NS >= 1 && NS <= kSlots, "frontier slots");
  unsigned long long fkey[NS];
  uint32_t ftie[NS];
  NodeRecs rec;  // nodes lane, lane + 32, ...
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    fkey[k] = 0ull;
    ftie[k] = kInvalid;
  }
  if (lane == 0 && !bad && budget > 0) {
    fkey[0] = score_key(0.0 + s_logp[0]);  // the root's first child: (1, 0, 0)
    ftie[0] = tie_of(1, 0, 0, kNoPrev);
  }
  unsigned long long bkey = fkey[0];  // this lane's best entry
  uint32_t btie = ftie[0];
  int bslot = 0;

  int n = 1;
  int used = 1;  // frontier positions handed out so far (positions are reused)
  for (; n < Q && !bad; ++n) {
    __syncwarp();  // node scores written by earlier pops are visible
    // warp argmax in three hardware reductions: key high word, low word, tie
    const bool valid = btie != kInvalid;
    const uint32_t hi = valid ? (uint32_t)(bkey >> 32) : 0u;
    const uint32_t m1 = __reduce_max_sync(0xffffffffu, hi);
    const bool c1 = valid && hi == m1;
    const uint32_t m2 = __reduce_max_sync(0xffffffffu, c1 ? (uint32_t)bkey : 0u);
    const bool c2 = c1 && (uint32_t)bkey == m2;
    const uint32_t m3 = __reduce_min_sync(0xffffffffu, c2 ? btie : kInvalid);
    if (m3 == kInvalid) break;  // candidate tree exhausted
    const bool winner = c2 && btie == m3;

    const double ps = key_score(((unsigned long long)m1 << 32) | m2);
    const int d = (int)(m3 >> 24);
    const int r = (int)((m3 >> 16) & 0xFFu);
    const int par = (int)((m3 >> 8) & 0xFFu);
    if (lane == (n & 31)) {  // record node n
      rec.set(n >> 5, m3);
      S.score[n] = ps;
    }

    // The popped entry's position takes the first push (its child, else its
    // next sibling), a new position `used` the second (the sibling). Only the
    // lanes that store a push add its score, with ONE double add between
    // them: GB300's FP64 pipe spends ~64 cycles on a double add however few
    // lanes are active, and two adds serialise.
    const bool has_child = d < De;   // rank 0 one level down
    const bool has_sib = r + 1 < Ke;  // next rank under the same parent
    const bool two = has_child && has_sib;
    const bool takes_second = two && lane == (used & 31);
    const uint32_t ct = tie_of(d + 1, 0, n, kNoPrev);
    const uint32_t st = tie_of(d, r + 1, par, (uint32_t)n);
    const int ci = has_child ? d * Ke : 0;              // (d+1, 0)
    const int si = has_sib ? (d - 1) * Ke + r + 1 : 0;  // (d, r+1)
    unsigned long long k1 = 0ull, k2 = 0ull;
    if (winner || takes_second) {
      const bool child_here = winner && has_child;  // this lane adds the child's score
      const double base = child_here ? ps : S.score[par];
      const unsigned long long kx = score_key(base + s_logp[child_here ? ci : si]);
      k1 = kx;
      k2 = kx;
      if (child_here && takes_second) k2 = score_key(S.score[par] + s_logp[si]);  // rare
    }
    const uint32_t t1 = has_child ? ct : (has_sib ? st : kInvalid);
    const int ns = used >> 5;

    // branch-free update of this lane's slots; its best entry by a
    // comparison tree
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const bool w1 = winner && k == bslot;
      const bool w2 = takes_second && k == ns;
      fkey[k] = w1 ? k1 : (w2 ? k2 : fkey[k]);
      ftie[k] = w1 ? t1 : (w2 ? st : ftie[k]);
    }
    if constexpr (NS == 1) {
      bkey = fkey[0];
      btie = ftie[0];
      bslot = 0;
    } else {
      const bool b01 = before(fkey[1], ftie[1], fkey[0], ftie[0]);
      const unsigned long long ka = b01 ? fkey[1] : fkey[0];
      const uint32_t ta = b01 ? ftie[1] : ftie[0];
      const int sa = b01 ? 1 : 0;
      if constexpr (NS == 2) {
        bkey = ka;
        btie = ta;
        bslot = sa;
      } else {
        unsigned long long kb = fkey[2];
        uint32_t tb = ftie[2];
        int sb = 2;
        if constexpr (NS == 4) {
          const bool b23 = before(fkey[3], ftie[3], fkey[2], ftie[2]);
          kb = b23 ? fkey[3] : fkey[2];
          tb = b23 ? ftie[3] : ftie[2];
          sb = b23 ? 3 : 2;
        }
        const bool bab = before(kb, tb, ka, ta);
        bkey = bab ? kb : ka;
        btie = bab ? tb : ta;
        bslot = bab ? sb : sa;
      }
    }
    if (two) ++used;
  }
  const int n_nodes = bad ? 1 : n;

  // ---- node records -> parents, depths, tokens, child links -----------------
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int c = lane + 32 * k;
    const uint32_t m = rec.tie(k);
    if (c >= Q) {
    } else if (c == 0) {
      S.par[0] = -1;
      S.dep[0] = 0;
      S.tok[0] = root;
    } else if (c < n_nodes) {
      const int d = (int)(m >> 24), r = (int)((m >> 16) & 0xFFu), p = (int)((m >> 8) & 0xFFu);
      S.par[c] = p;
      S.dep[c] = d;
      S.tok[c] = s_ids[(d - 1) * Ke + r];
      if (r == 0) S.fc[p] = c;
      else S.ns[m & 0xFFu] = c;
    } else {
      S.par[c] = -1;
      S.dep[c] = -1;
      S.tok[c] = 0;
    }
  }
  __syncwarp();
  // ---- ancestor words: own bit plus every node on the path to the root ------
  static_assert(kMaxW == 2, "ancestor words");
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int c = lane + 32 * k;
    if (c < Q) {
      unsigned long long w0 = 0ull, w1 = 0ull;
      int a = c;
      while (a >= 0) {
        if (a < 64) w0 |= 1ull << a;
        else w1 |= 1ull << (a - 64);
        a = (c < n_nodes) ? S.par[a] : -1;
      }
      S.anc[c][0] = w0;
      S.anc[c][1] = w1;
    }
  }
  __syncwarp();
  *bad_out = bad;
  return n_nodes;
}

// Writes the tree of sequence b from S (filled by build_warp) with the calling
// warp: tokens, parents, depths, vis_bits [Q][W], optional dense vis [Q][Q],
// first_child, next_sibling, n_nodes. Returns the status bits of the build.
__device__ __forceinline__ int32_t write_warp(const Smem& S, int b, int Q, int n_nodes, bool bad,
                                              int32_t* tokens, int32_t* parents, int32_t* depths,
                                              unsigned long long* vis_bits, uint8_t* vis,
                                              int32_t* first_child, int32_t* next_sibling,
                                              int32_t* n_nodes_out) {
  const int lane = threadIdx.x & 31;
  const int W = (Q + 63) / 64;
  int32_t* tok_o = tokens + (size_t)b * Q;
  int32_t* par_o = parents + (size_t)b * Q;
  int32_t* dep_o = depths + (size_t)b * Q;
  int32_t* fc_o = first_child + (size_t)b * Q;
  int32_t* ns_o = next_sibling + (size_t)b * Q;
  unsigned long long* vb_o = vis_bits + (size_t)b * Q * W;
  for (int c = lane; c < Q; c += 32) {
    tok_o[c] = S.tok[c];
    par_o[c] = S.par[c];
    dep_o[c] = S.dep[c];
    fc_o[c] = S.fc[c];
    ns_o[c] = S.ns[c];
    for (int w = 0; w < W; ++w) vb_o[(size_t)c * W + w] = S.anc[c][w];
  }
  if (vis != nullptr) {
    uint8_t* v_o = vis + (size_t)b * Q * Q;
    for (int e = lane; e < Q * Q; e += 32) {
      const int c = e / Q, j = e % Q;
      v_o[e] = (uint8_t)((S.anc[c][j >> 6] >> (j & 63)) & 1ull);
    }
  }
  if (lane == 0) n_nodes_out[b] = n_nodes;
  int32_t st = 0;
  if (bad) st |= DDT_ST_INPUT;
  if (n_nodes < Q) st |= DDT_ST_BUDGET_PAD;
  return st;
}

}  // namespace tb
}  // namespace ddt
