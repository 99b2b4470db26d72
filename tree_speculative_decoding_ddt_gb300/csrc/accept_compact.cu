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
// One CTA per sequence. Warp 0 walks the tree: every lane holds four tree
// slots in registers, one ballot per 32 slots finds the lowest-slot child
// whose token matches the target argmax. Then all threads move 16-byte
// chunks.
#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 256;
constexpr int kSlotsPerLane = kMaxQ / 32;

__global__ void __launch_bounds__(kThreads) k_accept_compact(AcceptCompactArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int32_t s_path[kMaxQ + 1];
  __shared__ int32_t s_len;
  __shared__ int32_t s_status;
  __shared__ int32_t s_target[kMaxQ];

  // a kernel launched as this one's programmatic dependent (the split-KV
  // merge of the same step) needs nothing from it: let it start now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int D = a.D;

  if (a.do_accept) {
    const int Q = a.Q;
    for (int c = tid; c < Q; c += kThreads) s_target[c] = a.target[(size_t)b * Q + c];
    __syncthreads();
    if (warp == 0) {
      int32_t tok[kSlotsPerLane], par[kSlotsPerLane];
#pragma unroll
      for (int k = 0; k < kSlotsPerLane; ++k) {
        const int c = lane + 32 * k;
        tok[k] = c < Q ? a.tokens[(size_t)b * Q + c] : 0;
        par[k] = c < Q ? a.parents[(size_t)b * Q + c] : -2;
      }
      unsigned long long visited_lo = 1ull, visited_hi = 0ull;  // slot 0 (root) is on the path
      int cur = 0, len = 0, st = 0;
      if (lane == 0) s_path[0] = 0;
      for (int hop = 0; hop < D; ++hop) {
        const int32_t want = s_target[cur];
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
        if (lane == 0) s_path[len] = nxt;
        cur = nxt;
      }
      __syncwarp();
      const int32_t bonus = s_target[cur];
      int32_t* idx_o = a.accept_idx + (size_t)b * (D + 1);
      int32_t* tok_o = a.out_tokens + (size_t)b * (D + 1);
      for (int d = lane; d <= D; d += 32) {
        const int slot = d <= len ? s_path[d] : -1;
        idx_o[d] = slot;
        int32_t t = -1;
        if (d < len) t = a.tokens[(size_t)b * Q + s_path[d + 1]];
        else if (d == len) t = bonus;
        tok_o[d] = t;
      }
      if (lane == 0) {
        a.accept_len[b] = len;
        a.bonus[b] = bonus;
        s_len = len;
        s_status = st;
      }
    }
    __syncthreads();
  } else {
    if (tid == 0) {
      int len = a.accept_len[b];
      s_len = len;
      s_status = 0;
    }
    __syncthreads();
    const int len = s_len;
    for (int d = tid; d <= D && d <= len && len >= 0; d += kThreads)
      s_path[d] = a.accept_idx[(size_t)b * (D + 1) + d];
    __syncthreads();
  }

  if (a.do_compact) {
    const int len = s_len;
    const int64_t L = a.prefix_len[b];
    const int64_t cap = (int64_t)a.max_pages * a.page_size;
    const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
    // validity of the whole path (identical decision in every thread)
    bool bad = len < 0 || len > D || L < 0 || L + len >= cap;
    if (!bad) {
      for (int d = 1; d <= len; ++d) {
        const int64_t i = s_path[d];
        if (i < 0 || L + i >= cap) bad = true;
      }
    }
    if (!bad) {
      for (int d = tid; d < 2 * len; d += kThreads) {
        const int64_t slot = d < len ? L + s_path[d + 1] : L + (d - len) + 1;
        const int64_t row = slot_row(bt, a.page_size, slot);
        if (row < 0 || row >= a.kv_rows) bad = true;
      }
      bad = __syncthreads_or(bad);
    }
    if (bad) {
      if (tid == 0) {
        a.new_len[b] = (int32_t)L;
        a.status[b] |= s_status | DDT_ST_RANGE;
      }
      return;
    }
    const int chunks_per_row = a.row_bytes / 16;
    const int total = len * chunks_per_row;
    uint4* buf = reinterpret_cast<uint4*>(smem_raw);
    for (int e = tid; e < total; e += kThreads) {
      const int d = e / chunks_per_row + 1, ch = e % chunks_per_row;
      const int64_t row = slot_row(bt, a.page_size, L + s_path[d]);
      buf[e] = reinterpret_cast<const uint4*>(a.kv + row * a.row_bytes)[ch];
    }
    __syncthreads();
    for (int e = tid; e < total; e += kThreads) {
      const int d = e / chunks_per_row + 1, ch = e % chunks_per_row;
      const int64_t row = slot_row(bt, a.page_size, L + d);
      reinterpret_cast<uint4*>(a.kv + row * a.row_bytes)[ch] = buf[e];
    }
    if (tid == 0) {
      a.new_len[b] = (int32_t)(L + 1 + len);
      a.status[b] |= s_status;
    }
  } else if (tid == 0) {
    a.status[b] |= s_status;
  }
}

}  // namespace

size_t accept_compact_smem_bytes(int32_t D, int32_t row_bytes) {
  return (size_t)D * (size_t)row_bytes;
}

cudaError_t launch_accept_compact(const AcceptCompactArgs& a, cudaStream_t stream) {
  const size_t smem = a.do_compact ? accept_compact_smem_bytes(a.D, a.row_bytes) : 0;
  static int smem_set[64] = {};
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit(k_accept_compact, (int)smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  k_accept_compact<<<a.B, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ddt
