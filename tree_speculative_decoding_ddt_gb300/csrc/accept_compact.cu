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
// gather/copy rows). The accepted rows are first read into shared memory by
// the whole CTA and only then written, so a source slot that is also a
// later destination slot is read before it is overwritten.
//
// A CTA serves up to eight sequences (one per warp; one per CTA when the
// batch is small, so every thread helps with one sequence's rows). A warp
// walks its tree: every lane holds four tree slots in registers, one ballot
// per 32 slots finds the lowest-slot child whose token matches the target
// argmax. Then all threads of the CTA move the accepted rows of all its
// sequences in 16-byte chunks: every row into shared memory, a barrier, every
// row out.
#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlotsPerLane = kMaxQ / 32;

// seqs: sequences per CTA (1..kWarps); sequence blockIdx.x * seqs + w is
// walked by warp w. The dynamic shared memory holds seqs x D rows.
__global__ void __launch_bounds__(kThreads) k_accept_compact(AcceptCompactArgs a, int seqs) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int32_t s_path[kWarps][kMaxQ + 1];
  __shared__ int32_t s_len[kWarps];
  __shared__ int32_t s_status[kWarps];
  __shared__ int32_t s_ok[kWarps];

  // a kernel launched as this one's programmatic dependent (the split-KV
  // merge of the same step) needs nothing from it: let it start now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int D = a.D;
  const int Q = a.Q;
  const long long b0 = (long long)blockIdx.x * seqs;

  if (warp < seqs) {
    const long long b = b0 + warp;
    if (b >= a.B) {
      if (lane == 0) s_len[warp] = -1;
    } else if (a.do_accept) {
      int32_t tok[kSlotsPerLane], par[kSlotsPerLane], tgt[kSlotsPerLane];
#pragma unroll
      for (int k = 0; k < kSlotsPerLane; ++k) {
        const int c = lane + 32 * k;
        tok[k] = c < Q ? a.tokens[b * Q + c] : 0;
        par[k] = c < Q ? a.parents[b * Q + c] : -2;
        tgt[k] = c < Q ? a.target[b * Q + c] : 0;
      }
      // target argmax at slot c, from the lane that holds it
      auto target_at = [&](int c) -> int32_t {
        int32_t v = tgt[0];
#pragma unroll
        for (int k = 1; k < kSlotsPerLane; ++k)
          if ((c >> 5) == k) v = tgt[k];
        return __shfl_sync(0xffffffffu, v, c & 31);
      };
      unsigned long long visited_lo = 1ull, visited_hi = 0ull;  // slot 0 (root) is on the path
      int cur = 0, len = 0, st = 0;
      if (lane == 0) s_path[warp][0] = 0;
      for (int hop = 0; hop < D; ++hop) {
        const int32_t want = target_at(cur);
        int nxt = -1;
#pragma unroll
        for (int k = 0; k < kSlotsPerLane; ++k) {
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
      const int32_t bonus = target_at(cur);
      __syncwarp();
      int32_t* idx_o = a.accept_idx + b * (D + 1);
      int32_t* tok_o = a.out_tokens + b * (D + 1);
      for (int d = lane; d <= D; d += 32) {
        const int slot = d <= len ? s_path[warp][d] : -1;
        idx_o[d] = slot;
        int32_t t = -1;
        if (d < len) t = a.tokens[b * Q + s_path[warp][d + 1]];
        else if (d == len) t = bonus;
        tok_o[d] = t;
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
      }
      for (int d = lane; d <= D && d <= len && len >= 0; d += 32)
        s_path[warp][d] = a.accept_idx[b * (D + 1) + d];
    }
  }
  __syncthreads();

  if (!a.do_compact) {
    if (warp < seqs && lane == 0 && b0 + warp < a.B) a.status[b0 + warp] |= s_status[warp];
    return;
  }
  // validity of every path (warp w decides for its sequence)
  if (warp < seqs) {
    const long long b = b0 + warp;
    const int len = s_len[warp];
    bool bad = true;
    if (b < a.B) {
      const int64_t L = a.prefix_len[b];
      const int64_t cap = (int64_t)a.max_pages * a.page_size;
      const int32_t* bt = a.block_table + b * a.max_pages;
      bad = len < 0 || len > D || L < 0 || L + len >= cap;
      if (!bad) {
        for (int d = 1 + lane; d <= len; d += 32) {
          const int64_t i = s_path[warp][d];
          if (i < 0 || L + i >= cap) bad = true;
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      if (!bad) {
        for (int d = lane; d < 2 * len; d += 32) {
          const int64_t slot = d < len ? L + s_path[warp][d + 1] : L + (d - len) + 1;
          const int64_t row = slot_row(bt, a.page_size, slot);
          if (row < 0 || row >= a.kv_rows) bad = true;
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      if (lane == 0) {
        if (bad) {
          a.new_len[b] = (int32_t)L;
          a.status[b] |= s_status[warp] | DDT_ST_RANGE;
        }
        s_ok[warp] = !bad;
      }
    } else if (lane == 0) {
      s_ok[warp] = 0;
    }
  }
  __syncthreads();
  // every accepted row of the CTA's sequences into shared memory, then out:
  // one flat range of 16-byte chunks over all of them, so every thread keeps
  // several loads in flight whatever the sequences' lengths
  const int chunks_per_row = a.row_bytes / 16;
  int off[kWarps + 1];  // first chunk of each sequence in the flat range
  off[0] = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    off[w + 1] = off[w] + ((w < seqs && s_ok[w]) ? s_len[w] * chunks_per_row : 0);
  const int total = off[kWarps];
  uint4* buf = reinterpret_cast<uint4*>(smem_raw);
  auto locate = [&](int e, int& w, int& d, int& ch) {
    w = 0;
#pragma unroll
    for (int k = 1; k < kWarps; ++k)
      if (e >= off[k]) w = k;
    const int r = e - off[w];
    d = r / chunks_per_row + 1;
    ch = r % chunks_per_row;
  };
  constexpr int kBatch = 4;  // loads a thread issues before storing any
  for (int e0 = tid; e0 < total; e0 += kThreads * kBatch) {
    uint4 v[kBatch];
    size_t at[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int e = e0 + k * kThreads;
      if (e >= total) break;
      int w, d, ch;
      locate(e, w, d, ch);
      const long long b = b0 + w;
      const int64_t row = slot_row(a.block_table + b * a.max_pages, a.page_size,
                                   (int64_t)a.prefix_len[b] + s_path[w][d]);
      v[k] = reinterpret_cast<const uint4*>(a.kv + row * a.row_bytes)[ch];
      at[k] = (size_t)w * D * chunks_per_row + (size_t)(d - 1) * chunks_per_row + ch;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (e0 + k * kThreads < total) buf[at[k]] = v[k];
  }
  __syncthreads();
  for (int e = tid; e < total; e += kThreads) {
    int w, d, ch;
    locate(e, w, d, ch);
    const long long b = b0 + w;
    const int64_t row = slot_row(a.block_table + b * a.max_pages, a.page_size,
                                 (int64_t)a.prefix_len[b] + d);
    reinterpret_cast<uint4*>(a.kv + row * a.row_bytes)[ch] =
        buf[(size_t)w * D * chunks_per_row + (size_t)(d - 1) * chunks_per_row + ch];
  }
  if (tid < seqs && s_ok[tid]) {
    const long long b = b0 + tid;
    a.new_len[b] = (int32_t)(a.prefix_len[b] + 1 + s_len[tid]);
    a.status[b] |= s_status[tid];
  }
}

}  // namespace

size_t accept_compact_smem_bytes(int32_t D, int32_t row_bytes) {
  return (size_t)D * (size_t)row_bytes;
}

cudaError_t launch_accept_compact(const AcceptCompactArgs& a, cudaStream_t stream) {
  // sequences per CTA: one while the batch leaves SMs free (every thread then
  // helps with that sequence's rows), up to eight (one per warp) beyond, as
  // many as the rows' shared memory allows
  const size_t per_seq = a.do_compact ? accept_compact_smem_bytes(a.D, a.row_bytes) : 0;
  int seqs = 1;
  if (a.B > 2LL * device_sm_count()) {
    seqs = kWarps;
    while (seqs > 1 && per_seq * (size_t)seqs > 200 * 1024) seqs /= 2;
  }
  const size_t smem = per_seq * (size_t)seqs;
  static int smem_set[64] = {};
  if (smem + sizeof(int32_t) * kWarps * (kMaxQ + 4) > 48 * 1024) {  // with the static arrays
    cudaError_t e = ensure_smem_limit(k_accept_compact, (int)smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  const long long grid = (a.B + seqs - 1) / seqs;
  k_accept_compact<<<(unsigned)grid, kThreads, smem, stream>>>(a, seqs);
  return cudaGetLastError();
}

}  // namespace ddt
