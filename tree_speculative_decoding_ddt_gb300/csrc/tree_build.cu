// A. Best-first draft-tree construction on the GPU.
//
// "The Milestone Commit: Cementing a Native DDTree Inference Engine",
// sections "What the Message Actually Does" and "The Reasoning Behind the
// Architecture": the builder replaces a CPU heapq, accumulates log-weights in
// double so that its pop order is bit-identical to the reference, keeps each
// node's ancestor set as a bitmask (parent mask | own bit) and emits the
// first-child / next-sibling encoding alongside tokens, parents and depths.
//
// GB300 layout: one warp per sequence. The frontier (at most budget+1 live
// entries, since every pop removes one entry and adds at most two) lives in
// registers, four entries per lane; each pop is a 32-lane argmax over
// (score desc, depth, rank, parent) done with three redux.sync reductions on
// integer keys, followed by two pushes. Node records (score, ancestors,
// child lists) stay in shared memory and are written out at the end.
//
// Two facts keep the shared-memory footprint small without changing the
// output: a node at depth d is popped at slot >= d, and a node of rank r at
// depth d at slot >= d + r, so pushes that can never be popped within the
// budget (depth or rank >= budget) are skipped; they could never be the
// frontier's best before the budget runs out.
#include <math.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr uint32_t kInvalid = 0xFFFFFFFFu;
constexpr int kSlots = kMaxQ / 32;  // frontier entries per lane

struct BuildShared {
  double n_score[kMaxQ];  // node scores
  int32_t n_tok[kMaxQ];
  int32_t n_par[kMaxQ];
  int32_t n_dep[kMaxQ];
  int32_t first_child[kMaxQ];
  int32_t next_sib[kMaxQ];
  int32_t last_child[kMaxQ];
  unsigned long long anc[kMaxQ][kMaxW];
};

// Order-preserving map of a double to a uint64: a larger score gives a larger
// key, -0.0 and +0.0 give the same key (they compare equal as doubles).
// GB300's FP64 pipe is narrow, so all heap comparisons run on these integer
// keys; only the two score additions per pop stay in FP64 (they must round
// exactly like the reference's double additions).
__device__ __forceinline__ unsigned long long score_key(double s) {
  unsigned long long u = (unsigned long long)__double_as_longlong(s);
  if (u == 0x8000000000000000ull) u = 0ull;
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_score(unsigned long long k) {
  const unsigned long long u = (k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
  return __longlong_as_double((long long)u);
}
// pop order: larger key first, then smaller tie word (depth<<16|rank<<8|parent)
__device__ __forceinline__ bool before(unsigned long long ka, uint32_t ta, unsigned long long kb,
                                       uint32_t tb) {
  if (ta == kInvalid) return false;
  if (tb == kInvalid) return true;
  return ka > kb || (ka == kb && ta < tb);
}

__global__ void __launch_bounds__(32) k_tree_build(
    int B, int D, int K, int budget, int V, int De, int Ke, const float* __restrict__ topk_logp,
    const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ root_tok,
    int32_t* __restrict__ tokens, int32_t* __restrict__ parents, int32_t* __restrict__ depths,
    unsigned long long* __restrict__ vis_bits, uint8_t* __restrict__ vis,
    int32_t* __restrict__ first_child, int32_t* __restrict__ next_sibling,
    int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BuildShared& S = *reinterpret_cast<BuildShared*>(smem_raw);
  float* s_logp = reinterpret_cast<float*>(smem_raw + sizeof(BuildShared));  // [De][Ke]
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_logp + De * Ke);             // [De][Ke]

  const int b = blockIdx.x;
  const int lane = threadIdx.x;
  const int Q = budget + 1;
  const int W = (Q + 63) / 64;
  const float* lp = topk_logp + (size_t)b * D * K;
  const int32_t* ip = topk_ids + (size_t)b * D * K;

  // ---- input validation over all D*K candidates --------------------------
  bool bad = false;
  for (int e = lane; e < D * K; e += 32) {
    const float x = lp[e];
    const int32_t t = ip[e];
    bad |= !isfinite(x) || t < 0 || t >= V;
  }
  const int32_t root = root_tok[b];
  bad |= (root < 0 || root >= V);
  bad = warp_any(bad);

  // ---- stage the reachable part of the candidate table ---------------------
  for (int e = lane; e < De * Ke; e += 32) {
    const int d = e / Ke, r = e % Ke;
    s_logp[e] = lp[d * K + r];
    s_ids[e] = ip[d * K + r];
  }
  for (int p = lane; p < kMaxQ; p += 32) {
    S.first_child[p] = -1;
    S.next_sib[p] = -1;
    S.last_child[p] = -1;
  }
  if (lane == 0) {
    S.n_score[0] = 0.0;
    S.n_tok[0] = root;
    S.n_par[0] = -1;
    S.n_dep[0] = 0;
    for (int w = 0; w < kMaxW; ++w) S.anc[0][w] = (w == 0) ? 1ull : 0ull;
  }
  __syncwarp();

  // ---- frontier: position p lives in lane p % 32, slot p / 32 ---------------
  unsigned long long fkey[kSlots];
  uint32_t ftie[kSlots];
#pragma unroll
  for (int k = 0; k < kSlots; ++k) {
    fkey[k] = 0ull;
    ftie[k] = kInvalid;
  }
  if (lane == 0 && !bad && budget > 0) {
    fkey[0] = score_key(0.0 + (double)s_logp[0]);
    ftie[0] = (1u << 16) | (0u << 8) | 0u;
  }
  unsigned long long bkey = fkey[0];  // this lane's best entry
  uint32_t btie = ftie[0];
  int bslot = 0;

  int n = 1;
  int used = 1;  // frontier positions handed out so far (positions are reused)
  for (; n < Q && !bad; ++n) {
    // warp argmax in three hardware reductions: key high word, key low word, tie
    const bool valid = btie != kInvalid;
    const uint32_t hi = valid ? (uint32_t)(bkey >> 32) : 0u;
    const uint32_t m1 = __reduce_max_sync(0xffffffffu, hi);
    const bool c1 = valid && hi == m1;
    const uint32_t m2 = __reduce_max_sync(0xffffffffu, c1 ? (uint32_t)bkey : 0u);
    const bool c2 = c1 && (uint32_t)bkey == m2;
    const uint32_t m3 = __reduce_min_sync(0xffffffffu, c2 ? btie : kInvalid);
    if (m3 == kInvalid) break;  // candidate tree exhausted
    const bool winner = c2 && btie == m3;

    const unsigned long long pkey = ((unsigned long long)m1 << 32) | m2;
    const double ps = key_score(pkey);
    const int d = (int)(m3 >> 16);
    const int r = (int)((m3 >> 8) & 0xFFu);
    const int par = (int)(m3 & 0xFFu);

    // the two pushes (computed by every lane)
    const bool has_child = d < De;   // rank 0 one level down
    const bool has_sib = r + 1 < Ke;  // next rank under the same parent
    unsigned long long ck = 0ull, sk = 0ull;
    uint32_t ct = kInvalid, st = kInvalid;
    if (has_child) {
      ck = score_key(ps + (double)s_logp[d * Ke]);
      ct = ((uint32_t)(d + 1) << 16) | (uint32_t)n;
    }
    if (has_sib) {
      sk = score_key(S.n_score[par] + (double)s_logp[(d - 1) * Ke + r + 1]);
      st = ((uint32_t)d << 16) | ((uint32_t)(r + 1) << 8) | (uint32_t)par;
    }
    // first push takes the popped position, the second a new one
    const unsigned long long k1 = has_child ? ck : sk;
    const uint32_t t1 = has_child ? ct : st;
    const bool two = has_child && has_sib;
    if (winner) {
#pragma unroll
      for (int k = 0; k < kSlots; ++k)
        if (k == bslot) {
          fkey[k] = k1;
          ftie[k] = t1;
        }
    }
    if (two && lane == (used & 31)) {
      const int ns = used >> 5;
#pragma unroll
      for (int k = 0; k < kSlots; ++k)
        if (k == ns) {
          fkey[k] = sk;
          ftie[k] = st;
        }
    }
    if (winner || (two && lane == (used & 31))) {
      bkey = 0ull;
      btie = kInvalid;
#pragma unroll
      for (int k = 0; k < kSlots; ++k)
        if (before(fkey[k], ftie[k], bkey, btie)) {
          bkey = fkey[k];
          btie = ftie[k];
          bslot = k;
        }
    }
    if (two) ++used;

    // node bookkeeping (off the critical path of the next pop)
    if (lane == 0) {
      S.n_score[n] = ps;
      S.n_tok[n] = s_ids[(d - 1) * Ke + r];
      S.n_par[n] = par;
      S.n_dep[n] = d;
      for (int w = 0; w < kMaxW; ++w) S.anc[n][w] = S.anc[par][w];
      S.anc[n][n >> 6] |= 1ull << (n & 63);
      if (S.first_child[par] < 0) {
        S.first_child[par] = n;
      } else {
        S.next_sib[S.last_child[par]] = n;
      }
      S.last_child[par] = n;
    }
    __syncwarp();
  }
  const int n_nodes = bad ? 1 : n;
  __syncwarp();

  // ---- write the tree ------------------------------------------------------
  int32_t* tok_o = tokens + (size_t)b * Q;
  int32_t* par_o = parents + (size_t)b * Q;
  int32_t* dep_o = depths + (size_t)b * Q;
  int32_t* fc_o = first_child + (size_t)b * Q;
  int32_t* ns_o = next_sibling + (size_t)b * Q;
  unsigned long long* vb_o = vis_bits + (size_t)b * Q * W;
  for (int c = lane; c < Q; c += 32) {
    const bool live = c < n_nodes;
    tok_o[c] = live ? S.n_tok[c] : 0;
    par_o[c] = live ? S.n_par[c] : -1;
    dep_o[c] = live ? S.n_dep[c] : -1;
    fc_o[c] = live ? S.first_child[c] : -1;
    ns_o[c] = live ? S.next_sib[c] : -1;
    for (int w = 0; w < W; ++w) {
      unsigned long long word;
      if (live) word = S.anc[c][w];
      else word = (w == (c >> 6)) ? (1ull << (c & 63)) : 0ull;
      vb_o[(size_t)c * W + w] = word;
    }
  }
  if (vis != nullptr) {
    uint8_t* v_o = vis + (size_t)b * Q * Q;
    for (int e = lane; e < Q * Q; e += 32) {
      const int c = e / Q, j = e % Q;
      bool on;
      if (c < n_nodes) on = (S.anc[c][j >> 6] >> (j & 63)) & 1ull;
      else on = (j == c);
      v_o[e] = on ? 1 : 0;
    }
  }
  if (lane == 0) {
    n_nodes_out[b] = n_nodes;
    int st = 0;
    if (bad) st |= DDT_ST_INPUT;
    if (n_nodes < Q) st |= DDT_ST_BUDGET_PAD;
    status[b] = st;
  }
}

}  // namespace

cudaError_t launch_tree_build(const ddt_tree_dims& d, const float* topk_logp,
                              const int32_t* topk_ids, const int32_t* root_tok, int32_t* tokens,
                              int32_t* parents, int32_t* depths, uint64_t* vis_bits, uint8_t* vis,
                              int32_t* first_child, int32_t* next_sibling, int32_t* n_nodes,
                              int32_t* status, cudaStream_t stream) {
  const int De = d.D < d.budget ? d.D : d.budget;
  const int Ke = d.K < d.budget ? d.K : d.budget;
  const size_t smem = sizeof(BuildShared) + (size_t)De * Ke * (sizeof(float) + sizeof(int32_t));
  static int smem_set[64] = {};
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit(k_tree_build, (int)smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  k_tree_build<<<d.B, 32, smem, stream>>>(
      d.B, d.D, d.K, d.budget, d.V, De, Ke, topk_logp, topk_ids, root_tok, tokens, parents,
      depths, reinterpret_cast<unsigned long long*>(vis_bits), vis, first_child, next_sibling,
      n_nodes, status);
  return cudaGetLastError();
}

}  // namespace ddt
