// Multi-step DDTree decode loop on the device: one CUDA graph whose single
// conditional WHILE node runs verify steps until every sequence has its
// tokens (or a step bound is reached), with no host round trip per step.
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": generate_ddtree wires tree_build -> verify_attn -> tree_accept +
// cache compaction with a drafter interface, and DDTree greedy output equals
// AR greedy output (the oracle drafter accepts 8.00 tokens per step: 3
// verify steps for 24 tokens). One step of the loop body, every call the
// library's own entry point:
//
//   drafter   k_loop_draft: the drafter's logits for depths 1..D (rows of a
//             per-position table, standing in for the drafter's forward)
//   top-K     ddt_drafter_topk
//   build     ddt_tree_build (root = the last committed token)
//   rope      ddt_rope_append (positions L + depth, tree latents to the cache)
//   attention ddt_verify_attn
//   target    k_loop_target: the target's logits at every tree slot (a
//             stream target standing in for the target's forward)
//   argmax    ddt_target_argmax
//   accept    accept + compaction (one kernel)
//   commit    k_loop_commit: append the accepted tokens and the bonus, move
//             the cache length, set the loop condition
//
// The synthetic drafter and target are the two model interfaces of the loop;
// everything else is the verify step itself.
#include <cuda_bf16.h>
#include <stdint.h>

#include <new>

#include "ddt_internal.cuh"

struct ddt_loop {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  ddt_loop_args args;
  int32_t* root_tok;
  int32_t* done;
  int32_t* loop_step;
};

namespace ddt {
namespace {

constexpr int kThreads = 256;
constexpr int kCommitThreads = 1024;

// Carving of the loop's workspace: every buffer 256-byte aligned.
struct LoopLayout {
  size_t drafter_logits, topk_logp, topk_ids, root_tok, tokens, parents, depths, first_child,
      next_sibling, n_nodes, vis_bits, q_rot, attn_out, lse, attn_ws, target_logits,
      target_argmax, accept_idx, accept_len, out_tokens, bonus, new_len, step_status, done,
      loop_step, total;
  size_t attn_ws_bytes;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

LoopLayout layout_of(const ddt_loop_args& a, size_t attn_ws_bytes) {
  const size_t B = a.tree.B, D = a.tree.D, K = a.tree.K, V = a.tree.V;
  const size_t Q = a.attn.Q, H = a.attn.H, C = a.attn.C, R = a.attn.R;
  const size_t W = (Q + 63) / 64;
  const size_t es = a.attn.dtype == DDT_BF16 ? 2 : 4;
  LoopLayout L{};
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t off = at;
    at += up256(bytes);
    return off;
  };
  L.drafter_logits = take(B * D * V * es);
  L.topk_logp = take(B * D * K * 4);
  L.topk_ids = take(B * D * K * 4);
  L.root_tok = take(B * 4);
  L.tokens = take(B * Q * 4);
  L.parents = take(B * Q * 4);
  L.depths = take(B * Q * 4);
  L.first_child = take(B * Q * 4);
  L.next_sibling = take(B * Q * 4);
  L.n_nodes = take(B * 4);
  L.vis_bits = take(B * Q * W * 8);
  L.q_rot = take(B * Q * H * R * es);
  L.attn_out = take(B * Q * H * C * es);
  L.lse = take(B * Q * H * 4);
  L.attn_ws = take(attn_ws_bytes);
  L.attn_ws_bytes = attn_ws_bytes;
  L.target_logits = take(B * Q * V * es);
  L.target_argmax = take(B * Q * 4);
  L.accept_idx = take(B * (D + 1) * 4);
  L.accept_len = take(B * 4);
  L.out_tokens = take(B * (D + 1) * 4);
  L.bonus = take(B * 4);
  L.new_len = take(B * 4);
  L.step_status = take(B * 4);
  L.done = take(B * 4);
  L.loop_step = take(4);
  L.total = at;
  return L;
}

__global__ void k_loop_init(int B, int G, int n_new, int max_steps,
                            const int32_t* __restrict__ golden,
                            const int32_t* __restrict__ prefix_len0, int32_t* prefix_len,
                            int32_t* committed, int32_t* n_committed, int32_t* steps,
                            int32_t* accepted, int32_t* status, int32_t* root_tok, int32_t* done,
                            int32_t* loop_step) {
  const int stride = gridDim.x * blockDim.x;
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  for (long long i = tid; i < (long long)B * (n_new + 1); i += stride) {
    const long long b = i / (n_new + 1), j = i % (n_new + 1);
    committed[i] = j == 0 ? golden[b * G] : -1;
  }
  for (long long i = tid; i < (long long)B * max_steps; i += stride) accepted[i] = 0;
  for (int b = tid; b < B; b += stride) {
    n_committed[b] = 1;
    steps[b] = 0;
    status[b] = 0;
    root_tok[b] = golden[(long long)b * G];
    prefix_len[b] = prefix_len0[b];
    done[b] = n_new == 0;
  }
  if (tid == 0) *loop_step = 0;
}

// Drafter logits: row (b, d) for d = 1..D is the table row of stream position
// n_b - 1 + d (n_b = tokens committed so far), clamped to the table.
__global__ void k_loop_draft(int B, int D, int G, long long row_bytes, int vec,
                             const uint8_t* __restrict__ table,
                             const int32_t* __restrict__ n_committed, uint8_t* __restrict__ out) {
  const long long unit = vec ? 16 : 2;
  const long long per_row = row_bytes / unit;
  const long long total = (long long)B * D * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / per_row, k = i % per_row;
    const int b = (int)(r / D), d = (int)(r % D) + 1;
    long long g = (long long)n_committed[b] - 1 + d;
    g = g < 0 ? 0 : (g > G - 1 ? G - 1 : g);
    const uint8_t* src = table + ((long long)b * G + g) * row_bytes;
    uint8_t* dst = out + r * row_bytes;
    if (vec)
      reinterpret_cast<uint4*>(dst)[k] = reinterpret_cast<const uint4*>(src)[k];
    else
      reinterpret_cast<uint16_t*>(dst)[k] = reinterpret_cast<const uint16_t*>(src)[k];
  }
}

// Target logits at tree slot s of sequence b: 1 at the target's greedy token,
// 0 elsewhere. The greedy token is the stream's next token when the slot's
// path from the root follows the stream, V-1 otherwise (and at padding
// slots).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    k_loop_target(int Q, long long V, int G, int vec, const int32_t* __restrict__ golden,
                  const int32_t* __restrict__ n_committed, const int32_t* __restrict__ tokens,
                  const int32_t* __restrict__ parents, const int32_t* __restrict__ depths,
                  T* __restrict__ logits) {
  __shared__ long long s_tgt;
  const int b = blockIdx.x / Q, s = blockIdx.x % Q;
  const int32_t* gb = golden + (long long)b * G;
  if (threadIdx.x == 0) {
    const long long n = n_committed[b];
    const int32_t* tk = tokens + (long long)b * Q;
    const int32_t* pa = parents + (long long)b * Q;
    const int32_t* de = depths + (long long)b * Q;
    const int dep = de[s];
    long long tgt = V - 1;
    if (dep >= 0) {
      bool ok = true;
      int c = s, hops = 0;
      while (c > 0 && c < Q && hops <= Q) {  // bounded walk to the root
        long long g = n - 1 + de[c];
        g = g < 0 ? 0 : (g > G - 1 ? G - 1 : g);
        if (tk[c] != gb[g]) ok = false;
        c = pa[c];
        ++hops;
      }
      if (c != 0) ok = false;
      if (ok && n + dep < G) tgt = gb[n + dep];
    }
    s_tgt = tgt;
  }
  __syncthreads();
  const long long tgt = s_tgt;
  T* row = logits + ((long long)b * Q + s) * V;
  if (vec) {
    constexpr int kPer = 16 / sizeof(T);
    const uint32_t one = sizeof(T) == 2 ? 0x3F80u : 0x3F800000u;  // 1.0
    for (long long v = threadIdx.x; v < V / kPer; v += blockDim.x) {
      uint4 w = make_uint4(0, 0, 0, 0);
      const long long j = tgt - v * kPer;
      if (j >= 0 && j < kPer) {
        uint32_t* p = reinterpret_cast<uint32_t*>(&w);
        if (sizeof(T) == 2)
          p[j / 2] = (j & 1) ? (one << 16) : one;
        else
          p[j] = one;
      }
      reinterpret_cast<uint4*>(row)[v] = w;
    }
  } else {
    for (long long v = threadIdx.x; v < V; v += blockDim.x)
      row[v] = (T)(v == tgt ? 1.0f : 0.0f);
  }
}

// Commit the step: the accepted drafts and the bonus join the sequence, the
// bonus is the next root, the cache length moves to the compacted length.
// A sequence whose step reported an error stops (its bits go to status).
// Last: continue the loop while a sequence is unfinished and the step bound
// is not reached.
__global__ void __launch_bounds__(kCommitThreads)
    k_loop_commit(int B, int D, int n_new, int max_steps, const int32_t* __restrict__ accept_len,
                  const int32_t* __restrict__ out_tokens, const int32_t* __restrict__ bonus,
                  const int32_t* __restrict__ new_len, const int32_t* __restrict__ step_status,
                  int32_t* committed, int32_t* n_committed, int32_t* steps, int32_t* accepted,
                  int32_t* status, int32_t* root_tok, int32_t* prefix_len, int32_t* done,
                  int32_t* loop_step, cudaGraphConditionalHandle handle) {
  bool active = false;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (done[b]) continue;
    const int st = step_status[b] & ~DDT_ST_BUDGET_PAD;
    if (st) {
      status[b] |= st;
      done[b] = 1;
      continue;
    }
    const int k = accept_len[b] + 1;
    const int n = n_committed[b];
    for (int i = 0; i < k; ++i)
      if (n + i < n_new + 1) committed[(long long)b * (n_new + 1) + n + i] = out_tokens[b * (D + 1) + i];
    n_committed[b] = n + k < n_new + 1 ? n + k : n_new + 1;
    const int s = steps[b];
    if (s < max_steps) accepted[(long long)b * max_steps + s] = k;
    steps[b] = s + 1;
    root_tok[b] = bonus[b];
    prefix_len[b] = new_len[b];
    if (n + k >= n_new + 1)
      done[b] = 1;
    else
      active = true;
  }
  const int any = __syncthreads_or(active);
  if (threadIdx.x == 0) {
    const int step = *loop_step + 1;
    *loop_step = step;
    cudaGraphSetConditional(handle, (any && step < max_steps) ? 1u : 0u);
  }
}

int check_loop(const ddt_loop_args* a) {
  if (a == nullptr) return DDT_EINVAL;
  const ddt_tree_dims& t = a->tree;
  const ddt_attn_dims& d = a->attn;
  if (t.B < 1 || t.D < 1 || t.K < 1 || t.budget < 0 || t.V < 2 || a->n_new < 0 ||
      a->max_steps < 1 || a->golden_len < 2)
    return DDT_EINVAL;
  if (d.B != t.B || d.Q != t.budget + 1) return DDT_EINVAL;
  if (d.dtype != DDT_BF16 && d.dtype != DDT_F32) return DDT_EINVAL;
  if (!a->golden || !a->drafter_table || !a->q_lat || !a->q_pe || !a->kv_new || !a->kv_cache ||
      !a->block_table || !a->prefix_len0 || !a->prefix_len || !a->committed ||
      !a->n_committed || !a->steps || !a->accepted || !a->status)
    return DDT_EINVAL;
  return DDT_OK;
}

#define DDT_TRY(x)              \
  do {                          \
    const int rc_ = (x);        \
    if (rc_ != DDT_OK) return rc_; \
  } while (0)
#define DDT_CUDA(x)                                   \
  do {                                                \
    if ((x) != cudaSuccess) return DDT_ELAUNCH;       \
  } while (0)

// Enqueue one verify step of the loop on `s` (inside the capture).
int enqueue_step(const ddt_loop_args& a, uint8_t* ws, const LoopLayout& L, int32_t* root_tok,
                 int32_t* done, int32_t* loop_step, cudaGraphConditionalHandle handle,
                 cudaStream_t s) {
  const ddt_tree_dims& t = a.tree;
  const ddt_attn_dims& d = a.attn;
  const int B = t.B, D = t.D, K = t.K, Q = d.Q;
  const long long V = t.V;
  const int es = d.dtype == DDT_BF16 ? 2 : 4;
  auto p32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  void* dl = ws + L.drafter_logits;
  float* tl = reinterpret_cast<float*>(ws + L.topk_logp);
  int32_t* tid = p32(L.topk_ids);
  int32_t* st = p32(L.step_status);

  // drafter
  {
    const long long row_bytes = V * es;
    const int vec = row_bytes % 16 == 0 &&
                    (reinterpret_cast<uintptr_t>(a.drafter_table) & 15u) == 0;
    const long long units = (long long)B * D * (row_bytes / (vec ? 16 : 2));
    const long long blocks = (units + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(blocks < 8LL * device_sm_count() ? blocks
                                                                      : 8LL * device_sm_count());
    k_loop_draft<<<grid, kThreads, 0, s>>>(B, D, a.golden_len, row_bytes, vec,
                                           static_cast<const uint8_t*>(a.drafter_table),
                                           a.n_committed, static_cast<uint8_t*>(dl));
    DDT_CUDA(cudaGetLastError());
  }
  DDT_TRY(ddt_drafter_topk((int64_t)B * D, V, K, d.dtype, dl, tl, tid, s));
  DDT_TRY(ddt_tree_build(&t, tl, tid, root_tok, p32(L.tokens), p32(L.parents), p32(L.depths),
                         reinterpret_cast<uint64_t*>(ws + L.vis_bits), nullptr,
                         p32(L.first_child), p32(L.next_sibling), p32(L.n_nodes), st, s));
  DDT_TRY(ddt_rope_append(&d, a.theta, p32(L.depths), a.prefix_len, a.block_table, a.q_pe,
                          ws + L.q_rot, a.kv_new, a.kv_cache, st, s));
  DDT_TRY(ddt_verify_attn(&d, a.q_lat, ws + L.q_rot, a.kv_cache, a.block_table, a.prefix_len,
                          reinterpret_cast<const uint64_t*>(ws + L.vis_bits), ws + L.attn_out,
                          reinterpret_cast<float*>(ws + L.lse), st,
                          L.attn_ws_bytes ? ws + L.attn_ws : nullptr, L.attn_ws_bytes, s));
  // target
  {
    void* lg = ws + L.target_logits;
    const int vec = (V * es) % 16 == 0;
    if (d.dtype == DDT_BF16)
      k_loop_target<__nv_bfloat16><<<(unsigned)((long long)B * Q), kThreads, 0, s>>>(
          Q, V, a.golden_len, vec, a.golden, a.n_committed, p32(L.tokens), p32(L.parents),
          p32(L.depths), static_cast<__nv_bfloat16*>(lg));
    else
      k_loop_target<float><<<(unsigned)((long long)B * Q), kThreads, 0, s>>>(
          Q, V, a.golden_len, vec, a.golden, a.n_committed, p32(L.tokens), p32(L.parents),
          p32(L.depths), static_cast<float*>(lg));
    DDT_CUDA(cudaGetLastError());
    DDT_TRY(ddt_target_argmax((int64_t)B * Q, V, d.dtype, lg, p32(L.target_argmax), s));
  }
  // accept + compaction
  {
    AcceptCompactArgs c{};
    c.B = B;
    c.Q = Q;
    c.D = D;
    c.do_accept = true;
    c.do_compact = true;
    c.tokens = p32(L.tokens);
    c.parents = p32(L.parents);
    c.target = p32(L.target_argmax);
    c.accept_idx = p32(L.accept_idx);
    c.accept_len = p32(L.accept_len);
    c.out_tokens = p32(L.out_tokens);
    c.bonus = p32(L.bonus);
    c.row_bytes = (d.C + d.R) * es;
    c.page_size = d.page_size;
    c.max_pages = d.max_pages;
    c.kv_rows = d.kv_rows;
    c.kv = static_cast<uint8_t*>(a.kv_cache);
    c.block_table = a.block_table;
    c.prefix_len = a.prefix_len;
    c.new_len = p32(L.new_len);
    c.status = st;
    DDT_CUDA(launch_accept_compact(c, s));
  }
  k_loop_commit<<<1, kCommitThreads, 0, s>>>(
      B, D, a.n_new, a.max_steps, p32(L.accept_len), p32(L.out_tokens), p32(L.bonus),
      p32(L.new_len), st, a.committed, a.n_committed, a.steps, a.accepted, a.status, root_tok,
      a.prefix_len, done, loop_step, handle);
  DDT_CUDA(cudaGetLastError());
  return DDT_OK;
}

}  // namespace
}  // namespace ddt

extern "C" {

size_t ddt_loop_workspace_size(const ddt_loop_args* a) {
  if (ddt::check_loop(a) != DDT_OK) return 0;
  return ddt::layout_of(*a, ddt_verify_attn_workspace_size(&a->attn)).total;
}

int ddt_loop_create(const ddt_loop_args* a, ddt_loop** out) {
  if (out == nullptr) return DDT_EINVAL;
  *out = nullptr;
  int rc = ddt::check_loop(a);
  if (rc) return rc;
  const ddt::LoopLayout L = ddt::layout_of(*a, ddt_verify_attn_workspace_size(&a->attn));
  if (a->workspace == nullptr || a->workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return DDT_EWORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);

  ddt_loop* h = new (std::nothrow) ddt_loop{};
  if (h == nullptr) return DDT_ELAUNCH;
  h->args = *a;
  h->root_tok = reinterpret_cast<int32_t*>(ws + L.root_tok);
  h->done = reinterpret_cast<int32_t*>(ws + L.done);
  h->loop_step = reinterpret_cast<int32_t*>(ws + L.loop_step);

  cudaStream_t cs = nullptr;
  rc = DDT_ELAUNCH;
  cudaGraphConditionalHandle cond = 0;
  cudaGraphNodeParams p = {};
  cudaGraphNode_t node = nullptr;
  cudaGraph_t body = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) goto fail;
  if (cudaGraphCreate(&h->graph, 0) != cudaSuccess) goto fail;
  if (cudaGraphConditionalHandleCreate(&cond, h->graph, 1, cudaGraphCondAssignDefault) !=
      cudaSuccess)
    goto fail;
  p.type = cudaGraphNodeTypeConditional;
  p.conditional.handle = cond;
  p.conditional.type = cudaGraphCondTypeWhile;
  p.conditional.size = 1;
  if (cudaGraphAddNode(&node, h->graph, nullptr, nullptr, 0, &p) != cudaSuccess) goto fail;
  body = p.conditional.phGraph_out[0];
  if (cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0,
                                    cudaStreamCaptureModeRelaxed) != cudaSuccess)
    goto fail;
  rc = ddt::enqueue_step(*a, ws, L, h->root_tok, h->done, h->loop_step, cond, cs);
  {
    cudaGraph_t captured = nullptr;
    const cudaError_t e = cudaStreamEndCapture(cs, &captured);
    if (rc == DDT_OK && e != cudaSuccess) rc = DDT_ELAUNCH;
  }
  if (rc != DDT_OK) goto fail;
  if (cudaGraphInstantiate(&h->exec, h->graph, 0) != cudaSuccess) {
    rc = DDT_ELAUNCH;
    goto fail;
  }
  cudaStreamDestroy(cs);
  *out = h;
  return DDT_OK;
fail:
  if (cs) cudaStreamDestroy(cs);
  if (h->graph) cudaGraphDestroy(h->graph);
  delete h;
  cudaGetLastError();  // leave no sticky launch error behind
  return rc == DDT_OK ? DDT_ELAUNCH : rc;
}

int ddt_loop_launch(ddt_loop* h, cudaStream_t stream) {
  if (h == nullptr) return DDT_EINVAL;
  const ddt_loop_args& a = h->args;
  ddt::k_loop_init<<<1, ddt::kThreads, 0, stream>>>(
      a.tree.B, a.golden_len, a.n_new, a.max_steps, a.golden, a.prefix_len0, a.prefix_len,
      a.committed, a.n_committed, a.steps, a.accepted, a.status, h->root_tok, h->done,
      h->loop_step);
  if (cudaGetLastError() != cudaSuccess) return DDT_ELAUNCH;
  return cudaGraphLaunch(h->exec, stream) == cudaSuccess ? DDT_OK : DDT_ELAUNCH;
}

int ddt_loop_destroy(ddt_loop* h) {
  if (h == nullptr) return DDT_OK;
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph) cudaGraphDestroy(h->graph);
  delete h;
  return DDT_OK;
}

}  // extern "C"
