// extern "C" entry points of libddt: host-side argument validation and
// dispatch to the kernels. Every function returns before the GPU work runs;
// see include/ddt.h for the contract of each call.
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace {

constexpr int kAbiVersion = 1;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tree_dims(const ddt_tree_dims* d) {
  if (d == nullptr) return DDT_EINVAL;
  if (d->B < 1 || d->D < 1 || d->K < 1 || d->budget < 0 || d->V < 1) return DDT_EINVAL;
  if (d->budget + 1 > DDT_MAX_Q) return DDT_EUNSUPPORTED;
  const int64_t De = d->D < d->budget ? d->D : d->budget;
  const int64_t Ke = d->K < d->budget ? d->K : d->budget;
  if (De * Ke > 8192) return DDT_EUNSUPPORTED;
  return DDT_OK;
}

int check_attn_dims(const ddt_attn_dims* d) {
  if (d == nullptr) return DDT_EINVAL;
  if (d->B < 1 || d->Q < 1 || d->H < 1 || d->C < 1 || d->R < 0 || d->page_size < 1 ||
      d->max_pages < 1 || d->kv_rows < 0 || !isfinite(d->scale))
    return DDT_EINVAL;
  if (d->Q > DDT_MAX_Q) return DDT_EUNSUPPORTED;
  if (d->dtype == DDT_F32) {
    if (d->C > 1024 || d->R > 256) return DDT_EUNSUPPORTED;
  } else if (d->dtype == DDT_BF16) {
    if (d->C != 512 || d->R != 64 || d->page_size % 64 != 0 || !(d->scale > 0.f))
      return DDT_EUNSUPPORTED;
  } else {
    return DDT_EINVAL;
  }
  return DDT_OK;
}

int check_accept(int32_t B, int32_t Q, int32_t D) {
  if (B < 1 || Q < 1 || D < 0) return DDT_EINVAL;
  if (Q > DDT_MAX_Q) return DDT_EUNSUPPORTED;
  return DDT_OK;
}

int check_compact(int32_t B, int32_t D, int32_t row_bytes, int32_t page_size, int32_t max_pages,
                  int64_t kv_rows, const void* kv) {
  if (B < 1 || D < 0 || row_bytes < 1 || page_size < 1 || max_pages < 1 || kv_rows < 0)
    return DDT_EINVAL;
  if (row_bytes % 16 != 0 || !aligned16(kv)) return DDT_EUNSUPPORTED;
  if (D > DDT_MAX_Q - 1) return DDT_EUNSUPPORTED;  // a path of a tree of at most DDT_MAX_Q slots
  return DDT_OK;
}

// The CUDA error behind the calling thread's most recent DDT_ELAUNCH.
thread_local int g_last_cuda_error = 0;
inline int launched(cudaError_t e) {
  if (e == cudaSuccess) return DDT_OK;
  g_last_cuda_error = (int)e;
  return DDT_ELAUNCH;
}

size_t attn_workspace(const ddt_attn_dims& d) {
  return d.dtype == DDT_BF16 ? ddt::verify_attn_bf16_workspace(d) : 0;
}

// Host-side checks of one verify-attention call that need the pointers.
int check_attn_call(const ddt_attn_dims* d, const void* q_lat, const void* q_pe, const void* kv,
                    const void* out, const void* ws, size_t ws_bytes) {
  if (d->dtype == DDT_F32) return DDT_OK;
  if (d->kv_rows < 1) return DDT_EINVAL;
  if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(kv) || !aligned16(out))
    return DDT_EUNSUPPORTED;
  const size_t need = attn_workspace(*d);
  if (need > 0 && (ws == nullptr || ws_bytes < need ||
                   (reinterpret_cast<uintptr_t>(ws) & 255u) != 0))
    return DDT_EWORKSPACE;
  return DDT_OK;
}

int run_attn(const ddt_attn_dims* d, const void* q_lat, const void* q_pe, const void* kv,
             const int32_t* block_table, const int32_t* prefix_len, const uint64_t* vis_bits,
             void* out, float* lse, int32_t* status, void* ws, size_t ws_bytes,
             cudaStream_t stream) {
  int rc = check_attn_call(d, q_lat, q_pe, kv, out, ws, ws_bytes);
  if (rc) return rc;
  if (d->dtype == DDT_F32) {
    return launched(ddt::launch_verify_attn_f32(
        *d, static_cast<const float*>(q_lat), static_cast<const float*>(q_pe),
        static_cast<const float*>(kv), block_table, prefix_len, vis_bits,
        static_cast<float*>(out), lse, status, stream));
  }
  return launched(ddt::launch_verify_attn_bf16(*d, q_lat, q_pe, kv, block_table, prefix_len,
                                               vis_bits, out, lse, status, ws, ws_bytes,
                                               stream));
}

}  // namespace

namespace ddt {
// SMs of the current device (cached per device).
int device_sm_count() {
  static int cached[64] = {};
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return n;
  if (cached[dev] == 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    cached[dev] = n;
  return cached[dev] ? cached[dev] : n;
}

// Host checks of a verify-attention call (dims, then pointers and alignment),
// shared with entry points defined in other files.
int check_verify_attn_args(const ddt_attn_dims* d, const void* q_lat, const void* q_pe,
                           const void* kv, const int32_t* block_table, const int32_t* prefix_len,
                           const uint64_t* vis_bits, const void* out, const int32_t* status) {
  int rc = check_attn_dims(d);
  if (rc) return rc;
  if (!q_lat || !q_pe || !kv || !block_table || !prefix_len || !vis_bits || !out || !status)
    return DDT_EINVAL;
  return DDT_OK;
}
}  // namespace ddt

extern "C" {

int ddt_abi_version(void) { return kAbiVersion; }

int ddt_last_cuda_error(void) { return g_last_cuda_error; }

int ddt_debug_checks(int* n_failed, int* first_site) {
  int (*const readers[])(int*) = {ddt::checks_read_pair,  ddt::checks_read_bf16,
                                  ddt::checks_read_f32,   ddt::checks_read_build,
                                  ddt::checks_read_accept, ddt::checks_read_rope,
                                  ddt::checks_read_topk,  ddt::checks_read_argmax};
  int total = 0, first = 0;
  for (auto rd : readers) {
    int f = 0;
    const int n = rd(&f);
    if (n > 0) {
      total += n;
      if (first == 0) first = f;
    }
  }
  if (n_failed) *n_failed = total;
  if (first_site) *first_site = first;
#ifdef DDT_CHECKS
  return 1;
#else
  return 0;
#endif
}

const char* ddt_cuda_error_name(int err) {
  return cudaGetErrorName(static_cast<cudaError_t>(err));
}

const char* ddt_strerror(int code) {
  switch (code) {
    case DDT_OK: return "ok";
    case DDT_EINVAL: return "invalid argument";
    case DDT_EUNSUPPORTED: return "unsupported dimensions, dtype or alignment";
    case DDT_ELAUNCH: return "CUDA launch failed";
    case DDT_EWORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown ddt error code";
  }
}

int ddt_tree_build(const ddt_tree_dims* dims, const float* topk_logp, const int32_t* topk_ids,
                   const int32_t* root_tok, int32_t* tokens, int32_t* parents, int32_t* depths,
                   uint64_t* vis_bits, uint8_t* vis, int32_t* first_child, int32_t* next_sibling,
                   int32_t* n_nodes, int32_t* status, cudaStream_t stream) {
  int rc = check_tree_dims(dims);
  if (rc) return rc;
  if (!topk_logp || !topk_ids || !root_tok || !tokens || !parents || !depths || !vis_bits ||
      !first_child || !next_sibling || !n_nodes || !status)
    return DDT_EINVAL;
  return launched(ddt::launch_tree_build(*dims, topk_logp, topk_ids, root_tok, tokens, parents,
                                         depths, vis_bits, vis, first_child, next_sibling,
                                         n_nodes, status, stream));
}

size_t ddt_verify_attn_workspace_size(const ddt_attn_dims* dims) {
  if (check_attn_dims(dims) != DDT_OK) return 0;
  return attn_workspace(*dims);
}

int ddt_verify_attn_rows_per_tile(const ddt_attn_dims* dims) {
  if (check_attn_dims(dims) != DDT_OK || dims->dtype != DDT_BF16) return 0;
  return ddt::verify_attn_bf16_rows_per_tile(*dims);
}

int ddt_verify_attn_splits(const ddt_attn_dims* dims) {
  if (check_attn_dims(dims) != DDT_OK || dims->dtype != DDT_BF16) return 0;
  return ddt::verify_attn_bf16_splits(*dims);
}

int ddt_verify_attn(const ddt_attn_dims* dims, const void* q_lat, const void* q_pe,
                    const void* kv_cache, const int32_t* block_table, const int32_t* prefix_len,
                    const uint64_t* vis_bits, void* out, float* lse, int32_t* status,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_attn_dims(dims);
  if (rc) return rc;
  if (!q_lat || !q_pe || !kv_cache || !block_table || !prefix_len || !vis_bits || !out || !status)
    return DDT_EINVAL;
  return run_attn(dims, q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits, out, lse,
                  status, workspace, workspace_bytes, stream);
}

int ddt_tree_accept(int32_t B, int32_t Q, int32_t D, const int32_t* tokens,
                    const int32_t* parents, const int32_t* target_argmax, int32_t* accept_idx,
                    int32_t* accept_len, int32_t* out_tokens, int32_t* bonus, int32_t* status,
                    cudaStream_t stream) {
  int rc = check_accept(B, Q, D);
  if (rc) return rc;
  if (!tokens || !parents || !target_argmax || !accept_idx || !accept_len || !out_tokens ||
      !bonus || !status)
    return DDT_EINVAL;
  ddt::AcceptCompactArgs a{};
  a.B = B; a.Q = Q; a.D = D;
  a.do_accept = true; a.do_compact = false;
  a.tokens = tokens; a.parents = parents; a.target = target_argmax;
  a.accept_idx = accept_idx; a.accept_len = accept_len; a.out_tokens = out_tokens;
  a.bonus = bonus; a.status = status;
  return launched(ddt::launch_accept_compact(a, stream));
}

int ddt_cache_compact(int32_t B, int32_t D, int32_t row_bytes, int32_t page_size,
                      int32_t max_pages, int64_t kv_rows, void* kv_cache,
                      const int32_t* block_table, const int32_t* prefix_len,
                      const int32_t* accept_idx, const int32_t* accept_len, int32_t* new_len,
                      int32_t* status, cudaStream_t stream) {
  if (!kv_cache || !block_table || !prefix_len || !accept_idx || !accept_len || !new_len ||
      !status)
    return DDT_EINVAL;
  int rc = check_compact(B, D, row_bytes, page_size, max_pages, kv_rows, kv_cache);
  if (rc) return rc;
  ddt::AcceptCompactArgs a{};
  a.B = B; a.D = D; a.Q = 1;
  a.do_accept = false; a.do_compact = true;
  a.accept_idx = const_cast<int32_t*>(accept_idx);
  a.accept_len = const_cast<int32_t*>(accept_len);
  a.row_bytes = row_bytes; a.page_size = page_size; a.max_pages = max_pages;
  a.kv_rows = kv_rows; a.kv = static_cast<uint8_t*>(kv_cache);
  a.block_table = block_table; a.prefix_len = prefix_len; a.new_len = new_len;
  a.status = status;
  return launched(ddt::launch_accept_compact(a, stream));
}

int ddt_target_argmax(int64_t rows, int64_t V, int dtype, const void* logits, int32_t* argmax,
                      cudaStream_t stream) {
  if (!logits || !argmax || rows < 1 || V < 1) return DDT_EINVAL;
  if (dtype != DDT_BF16 && dtype != DDT_F32) return DDT_EINVAL;
  if (rows > (int64_t(1) << 28) - 1 || V > 0x7fffffffLL) return DDT_EUNSUPPORTED;
  return launched(ddt::launch_target_argmax(rows, V, dtype, logits, argmax, stream));
}

int ddt_drafter_topk(int64_t rows, int64_t V, int32_t K, int dtype, const void* logits,
                     float* topk_logp, int32_t* topk_ids, cudaStream_t stream) {
  if (!logits || !topk_logp || !topk_ids || rows < 1 || V < 1 || K < 1) return DDT_EINVAL;
  if (dtype != DDT_BF16 && dtype != DDT_F32) return DDT_EINVAL;
  if (K > 16 || K > V || rows > (int64_t(1) << 28) - 1 || V > 0x7fffffffLL)
    return DDT_EUNSUPPORTED;
  return launched(ddt::launch_drafter_topk(rows, V, K, dtype, logits, topk_logp, topk_ids, stream));
}

int ddt_rope_append(const ddt_attn_dims* d, double theta, const int32_t* depths,
                    const int32_t* prefix_len, const int32_t* block_table, const void* q_pe_in,
                    void* q_pe_out, const void* kv_new, void* kv_cache, int32_t* status,
                    cudaStream_t stream) {
  if (d == nullptr || !depths || !prefix_len || !block_table || !q_pe_in || !q_pe_out || !kv_new ||
      !kv_cache || !status)
    return DDT_EINVAL;
  if (d->B < 1 || d->Q < 1 || d->H < 1 || d->C < 0 || d->R < 2 || d->R % 2 != 0 ||
      d->page_size < 1 || d->max_pages < 1 || d->kv_rows < 0 || !(theta > 0.0) ||
      !isfinite(theta))
    return DDT_EINVAL;
  if (d->dtype != DDT_BF16 && d->dtype != DDT_F32) return DDT_EINVAL;
  if (d->Q > DDT_MAX_Q || d->R / 2 > ddt::kMaxRopeHalf || (int64_t)d->B * d->Q > 0x7fffffffLL)
    return DDT_EUNSUPPORTED;
  ddt::RopeFreqs f = {};
  for (int i = 0; i < d->R / 2; ++i) f.f[i] = pow(theta, -2.0 * i / d->R);
  return launched(ddt::launch_rope_append(*d, f, depths, prefix_len, block_table, q_pe_in,
                                          q_pe_out, kv_new, kv_cache, status, stream));
}

size_t ddt_step_workspace_size(const ddt_step_args* args) {
  if (args == nullptr) return 0;
  return ddt_verify_attn_workspace_size(&args->attn);
}

int ddt_step(const ddt_step_args* a, cudaStream_t stream) {
  if (a == nullptr) return DDT_EINVAL;
  int rc = check_tree_dims(&a->tree);
  if (rc) return rc;
  rc = check_attn_dims(&a->attn);
  if (rc) return rc;
  if (a->tree.B != a->attn.B || a->attn.Q != a->tree.budget + 1) return DDT_EINVAL;
  const int elem = a->attn.dtype == DDT_BF16 ? 2 : 4;
  const int32_t row_bytes = (a->attn.C + a->attn.R) * elem;
  rc = check_compact(a->attn.B, a->tree.D, row_bytes, a->attn.page_size, a->attn.max_pages,
                     a->attn.kv_rows, a->kv_cache);
  if (rc) return rc;
  if (!a->topk_logp || !a->topk_ids || !a->root_tok || !a->q_lat || !a->q_pe || !a->kv_cache ||
      !a->block_table || !a->prefix_len || !a->target_argmax || !a->tokens || !a->parents ||
      !a->depths || !a->vis_bits || !a->first_child || !a->next_sibling || !a->n_nodes ||
      !a->out || !a->accept_idx || !a->accept_len || !a->out_tokens || !a->bonus ||
      !a->new_len || !a->status)
    return DDT_EINVAL;
  rc = check_attn_call(&a->attn, a->q_lat, a->q_pe, a->kv_cache, a->out, a->workspace,
                       a->workspace_bytes);
  if (rc) return rc;

  // C + D. accept and compaction in one kernel
  ddt::AcceptCompactArgs c{};
  c.B = a->attn.B; c.Q = a->attn.Q; c.D = a->tree.D;
  c.do_accept = true; c.do_compact = true;
  c.tokens = a->tokens; c.parents = a->parents; c.target = a->target_argmax;
  c.accept_idx = a->accept_idx; c.accept_len = a->accept_len; c.out_tokens = a->out_tokens;
  c.bonus = a->bonus;
  c.row_bytes = row_bytes; c.page_size = a->attn.page_size; c.max_pages = a->attn.max_pages;
  c.kv_rows = a->attn.kv_rows; c.kv = static_cast<uint8_t*>(a->kv_cache);
  c.block_table = a->block_table; c.prefix_len = a->prefix_len; c.new_len = a->new_len;
  c.status = a->status;

  const int64_t De = a->tree.D < a->tree.budget ? a->tree.D : a->tree.budget;
  const int64_t Ke = a->tree.K < a->tree.budget ? a->tree.K : a->tree.budget;
  if (a->attn.dtype == DDT_BF16 && De * Ke <= ddt::kFuseMaxCand) {
    // A inside B: the attention kernel builds the tree in a spare warp while
    // its prefix tiles run; status starts from zero and is OR-ed. C + D are
    // launched by the attention call, before its split-KV merge, which then
    // runs beside them
    if (cudaMemsetAsync(a->status, 0, sizeof(int32_t) * (size_t)a->attn.B, stream) != cudaSuccess)
      return DDT_ELAUNCH;
    ddt::TreeFuse f{};
    f.D = a->tree.D; f.K = a->tree.K; f.budget = a->tree.budget; f.V = a->tree.V;
    f.topk_logp = a->topk_logp; f.topk_ids = a->topk_ids; f.root_tok = a->root_tok;
    f.tokens = a->tokens; f.parents = a->parents; f.depths = a->depths;
    f.vis_bits = a->vis_bits; f.vis = a->vis; f.first_child = a->first_child;
    f.next_sibling = a->next_sibling; f.n_nodes = a->n_nodes;
    return launched(ddt::launch_verify_attn_bf16(a->attn, a->q_lat, a->q_pe, a->kv_cache,
                                                 a->block_table, a->prefix_len, a->vis_bits,
                                                 a->out, a->lse, a->status, a->workspace,
                                                 a->workspace_bytes, stream, &f, &c));
  }
  // A. build (overwrites status)
  if (ddt::launch_tree_build(a->tree, a->topk_logp, a->topk_ids, a->root_tok, a->tokens,
                             a->parents, a->depths, a->vis_bits, a->vis, a->first_child,
                             a->next_sibling, a->n_nodes, a->status, stream) != cudaSuccess)
    return DDT_ELAUNCH;
  // B. verify attention over the tree just built
  rc = run_attn(&a->attn, a->q_lat, a->q_pe, a->kv_cache, a->block_table, a->prefix_len,
                a->vis_bits, a->out, a->lse, a->status, a->workspace, a->workspace_bytes, stream);
  if (rc) return rc;
  return launched(ddt::launch_accept_compact(c, stream));
}

}  // extern "C"
