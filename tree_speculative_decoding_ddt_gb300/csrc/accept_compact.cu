// C. Greedy tree accept and D. post-verify cache compaction.
//
// Accept: "The Checkpoint: Committing a Working Native DDTree Engine",
// section "The Message" (tree_accept wired after verify_attn; DDTree greedy
// output must equal AR greedy output), and "The Milestone Commit", section
// "Mistakes and Incorrect Assumptions" (a crash of tree_accept on cyclic
// random data was fixed with a safety bound). Here the walk is bounded by D
// hops and stops with DDT_ST_CYCLE rather than revisiting a node.
//
// Compaction: "The Checkpoint", section "The Message" (cache append +
// post-verify compaction; after accept, gather the accepted-path latents;
// gather/copy rows). Row d of the path (slot s_d, d = 1..len) moves to slot d.
// Nodes are numbered in pop order, so a path from the root has strictly
// increasing slots, 0 = s_0 < s_1 < ... < s_len, hence s_d >= d: rows with
// s_d == d are already in place and are not touched, and for every moved row
// s_d > d. A moved row's destination d is never the source of a later row
// (those read slots s_d' >= d' > d), so rows copied in increasing d need no
// staging; only when some source slot is also a destination (s_d <= len) do
// the loads of a batch of rows wait at a barrier for all of them before the
// stores. A list that is not strictly increasing is not a path and is refused
// (DDT_ST_RANGE, sequence untouched).
//
// A CTA serves up to eight sequences (one per warp; one per CTA when the
// batch is small, so every thread helps with one sequence's rows). A warp
// walks its tree: every lane holds NSL tree slots in registers, one ballot
// per 32 slots finds the lowest-slot child whose token matches the target
// argmax. The warp then checks its path and lists the rows that move (byte
// offsets of source and destination); all threads of the CTA copy the listed
// rows of all its sequences as one flat range of 16-byte chunks, several
// loads in flight per thread.
#include "ddt_internal.cuh"

namespace ddt {
DDT_CHECKS_FILE(accept)
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 6;  // chunks a thread loads before storing any

// seqs: sequences per CTA (1..kWarps); sequence blockIdx.x * seqs + w is
// walked by warp w. NSL = ceil(Q / 32) tree slots per lane. kCompact: the
// compaction part is compiled in (a.do_compact); without it the kernel is
// small enough for eight CTAs per SM.
template <int NSL, bool kCompact>
__global__ void __launch_bounds__(kThreads, kCompact ? 4 : 8)
    k_accept_compact(AcceptCompactArgs a, int seqs) {
  __shared__ int32_t s_path[kWarps][kMaxQ + 1];
  __shared__ long long s_src[kWarps][kMaxQ];  // byte offsets of the moved rows' sources
  __shared__ long long s_dst[kWarps][kMaxQ];  // and destinations
  __shared__ int32_t s_len[kWarps];
  __shared__ int32_t s_status[kWarps];
  __shared__ int32_t s_moves[kWarps];  // rows that move (0 for a refused sequence)
  __shared__ int32_t s_hazard;

  // a kernel launched as this one's programmatic dependent (the split-KV
  // merge of the same step) needs nothing from it: let it start now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int D = a.D;
  const int Q = a.Q;
  const long long b0 = (long long)blockIdx.x * seqs;
  if (tid == 0) s_hazard = 0;

  if (warp < seqs) {
    const long long b = b0 + warp;
    if (b >= a.B) {
      if (lane == 0) s_len[warp] = -1;
    } else if (a.do_accept) {
      int32_t tok[NSL], par[NSL], tgt[NSL];
#pragma unroll
      for (int k = 0; k < NSL; ++k) {
        const int c = lane + 32 * k;
        tok[k] = c < Q ? a.tokens[b * Q + c] : 0;
        par[k] = c < Q ? a.parents[b * Q + c] : -2;
        tgt[k] = c < Q ? a.target[b * Q + c] : 0;
      }
      // value of a per-slot register array at slot c (the same c in every
      // lane), from the lane holding it
      auto at_slot = [&](const int32_t(&v)[NSL], int c) -> int32_t {
        int32_t x = v[0];
#pragma unroll
        for (int k = 1; k < NSL; ++k)
          if ((c >> 5) == k) x = v[k];
        return __shfl_sync(0xffffffffu, x, c & 31);
      };
      // the same with a slot of each lane's own
      auto at_lane_slot = [&](const int32_t(&v)[NSL], int c) -> int32_t {
        int32_t x = 0;
#pragma unroll
        for (int k = 0; k < NSL; ++k) {
          const int32_t y = __shfl_sync(0xffffffffu, v[k], c & 31);
          if ((c >> 5) == k) x = y;
        }
        return x;
      };
      unsigned long long visited_lo = 1ull, visited_hi = 0ull;  // slot 0 (root) is on the path
      int cur = 0, len = 0, st = 0;
      if (lane == 0) s_path[warp][0] = 0;
      for (int hop = 0; hop < D; ++hop) {
        const int32_t want = at_slot(tgt, cur);
        int nxt = -1;
#pragma unroll
        for (int k = 0; k < NSL; ++k) {
          const unsigned m = __ballot_sync(0xffffffffu, par[k] == cur && tok[k] == want);
          if (nxt < 0 && m) nxt = 32 * k + __ffs(m) - 1;
        }
        if (nxt < 0) break;
        const unsigned long long bit = 1ull << (nxt & 63);
        if (((nxt < 64) ? visited_lo : visited_hi) & bit) {
          st |= DDT_ST_CYCLE;
          break;
        }
        if (nxt < 64) visited_lo |= bit;
        else visited_hi |= bit;
        ++len;
        if (lane == 0) s_path[warp][len] = nxt;
        cur = nxt;
      }
      const int32_t bonus = at_slot(tgt, cur);
      __syncwarp();
      int32_t* idx_o = a.accept_idx + b * (D + 1);
      int32_t* tok_o = a.out_tokens + b * (D + 1);
      for (int d0 = 0; d0 <= D; d0 += 32) {  // every lane takes part in the shuffles
        const int d = d0 + lane;
        const int nxt_slot = d < len ? s_path[warp][d + 1] : 0;
        const int32_t t = at_lane_slot(tok, nxt_slot);  // token of the path's next node
        if (d <= D) {
          idx_o[d] = d <= len ? s_path[warp][d] : -1;
          tok_o[d] = d < len ? t : (d == len ? bonus : -1);
        }
      }
      if (lane == 0) {
        a.accept_len[b] = len;
        a.bonus[b] = bonus;
        s_len[warp] = len;
        s_status[warp] = st;
      }
    } else {
      const int len = a.accept_len[b];
      if (lane == 0) {
        s_len[warp] = len;
        s_status[warp] = 0;
        s_path[warp][0] = 0;  // the root; accept_idx[0] is not read
      }
      for (int d = 1 + lane; d <= D && d <= len; d += 32)
        s_path[warp][d] = a.accept_idx[b * (D + 1) + d];
    }
  }
  __syncthreads();

  if constexpr (!kCompact) {
    if (warp < seqs && lane == 0 && b0 + warp < a.B) a.status[b0 + warp] |= s_status[warp];
    return;
  }
  // each warp checks its sequence's path and lists the rows that move
  if (warp < seqs) {
    const long long b = b0 + warp;
    const int len = s_len[warp];
    int moves = 0;
    if (b < a.B) {
      const int64_t L = a.prefix_len[b];
      const int64_t cap = (int64_t)a.max_pages * a.page_size;
      const int32_t* bt = a.block_table + b * a.max_pages;
      bool bad = len < 0 || len > D || L < 0 || L + len >= cap;
      bool hazard = false;
      if (!bad) {
        // a path: 0 = s_0 < s_1 < ... < s_len, every slot inside the cache
        for (int d = 1 + lane; d <= len; d += 32) {
          const int64_t i = s_path[warp][d];
          if (i <= s_path[warp][d - 1] || L + i >= cap) bad = true;
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      if (!bad) {
        // rows of every source and destination slot inside the cache; the
        // moved ones listed in order of d
        for (int d0 = 1; d0 <= len; d0 += 32) {
          const int d = d0 + lane;
          bool mv = false;
          int64_t src = 0, dst = 0;
          if (d <= len) {
            const int64_t s = s_path[warp][d];
            src = slot_row(bt, a.page_size, L + s);
            dst = slot_row(bt, a.page_size, L + d);
            if (src < 0 || src >= a.kv_rows || dst < 0 || dst >= a.kv_rows) bad = true;
            mv = s != d;
            hazard |= mv && s <= len;  // a source that is also a destination
          }
          const unsigned m = __ballot_sync(0xffffffffu, mv);
          if (mv) {
            const int at = moves + __popc(m & ((1u << lane) - 1u));
            s_src[warp][at] = src * a.row_bytes;
            s_dst[warp][at] = dst * a.row_bytes;
          }
          moves += __popc(m);
        }
        bad = __any_sync(0xffffffffu, bad);
        hazard = __any_sync(0xffffffffu, hazard);
      }
      if (lane == 0) {
        if (bad) {
          a.new_len[b] = (int32_t)L;
          a.status[b] |= s_status[warp] | DDT_ST_RANGE;
        } else {
          a.new_len[b] = (int32_t)(L + 1 + len);
          a.status[b] |= s_status[warp];
          if (hazard) s_hazard = 1;
        }
        s_moves[warp] = bad ? 0 : moves;
      }
    } else if (lane == 0) {
      s_moves[warp] = 0;
    }
  }
  __syncthreads();
  // the listed rows of all the CTA's sequences as one flat range of 16-byte
  // chunks (sequence, then d, then chunk), in batches of kBatch chunks per
  // thread; consecutive batches follow increasing d within every sequence
  const int cpr = a.row_bytes >> 4;  // chunks per row
  int off[kWarps + 1];              // first flat row of each sequence
  off[0] = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) off[w + 1] = off[w] + (w < seqs ? s_moves[w] : 0);
  const long long total = (long long)off[kWarps] * cpr;
  const bool hazard = s_hazard != 0;
  // chunk e = tid + kThreads * j; its (flat row, chunk) advanced without division
  const int step_r = kThreads / cpr, step_c = kThreads % cpr;
  int r = tid / cpr, c = tid % cpr;
  for (long long e0 = 0; e0 < total; e0 += (long long)kThreads * kBatch) {
    uint4 v[kBatch];
    long long to[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      to[j] = -1;
      if (e0 + tid + (long long)kThreads * j < total) {
        int w = 0, first = 0;  // the sequence of flat row r and its first flat row
#pragma unroll
        for (int k = 1; k < kWarps; ++k)
          if (r >= off[k]) {
            w = k;
            first = off[k];
          }
        const int i = r - first;
        // both 16-byte pieces inside the cache (the slots were checked per row)
        const long long kv_bytes = a.kv_rows * (long long)a.row_bytes;
        if (DDT_GUARD(s_src[w][i] + 16 * c + 16 <= kv_bytes && s_dst[w][i] + 16 * c + 16 <= kv_bytes,
                      501, nullptr)) {
          v[j] = *reinterpret_cast<const uint4*>(a.kv + s_src[w][i] + 16 * c);
          to[j] = s_dst[w][i] + 16 * c;
        }
      }
      c += step_c;
      r += step_r;
      if (c >= cpr) {
        c -= cpr;
        ++r;
      }
    }
    if (hazard) __syncthreads();  // every source of this batch read before any write
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (to[j] >= 0) *reinterpret_cast<uint4*>(a.kv + to[j]) = v[j];
  }
}

template <int NSL>
void launch_k(const AcceptCompactArgs& a, int seqs, cudaStream_t stream) {
  const long long grid = (a.B + seqs - 1) / seqs;
  if (a.do_compact)
    k_accept_compact<NSL, true><<<(unsigned)grid, kThreads, 0, stream>>>(a, seqs);
  else
    k_accept_compact<NSL, false><<<(unsigned)grid, kThreads, 0, stream>>>(a, seqs);
}

}  // namespace

cudaError_t launch_accept_compact(const AcceptCompactArgs& a, cudaStream_t stream) {
  // sequences per CTA: one while the batch leaves SMs free (every thread then
  // helps with that sequence's rows), eight (one per warp) beyond
  const int seqs = a.B > 2LL * device_sm_count() ? kWarps : 1;
  const int nsl = a.do_accept ? (a.Q + 31) / 32 : 1;
  switch (nsl) {
    case 1: launch_k<1>(a, seqs, stream); break;
    case 2: launch_k<2>(a, seqs, stream); break;
    case 3: launch_k<3>(a, seqs, stream); break;
    default: launch_k<4>(a, seqs, stream); break;
  }
  return cudaGetLastError();
}

}  // namespace ddt
