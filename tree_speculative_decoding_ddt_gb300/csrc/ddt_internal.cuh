// Internal declarations shared by the translation units of libddt.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt.h"

namespace ddt {

constexpr int kMaxQ = DDT_MAX_Q;
constexpr int kMaxW = (kMaxQ + 63) / 64;

// ---- launchers (defined next to their kernels) ------------------------------

// A. tree build; validates nothing (the ABI layer does).
cudaError_t launch_tree_build(const ddt_tree_dims& d, const float* topk_logp,
                              const int32_t* topk_ids, const int32_t* root_tok, int32_t* tokens,
                              int32_t* parents, int32_t* depths, uint64_t* vis_bits, uint8_t* vis,
                              int32_t* first_child, int32_t* next_sibling, int32_t* n_nodes,
                              int32_t* status, cudaStream_t stream);

// C+D. Accept walk and/or compaction in one kernel (one CTA per sequence).
struct AcceptCompactArgs {
  int32_t B, Q, D;
  bool do_accept, do_compact;
  // accept
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* target;
  int32_t* accept_idx;  // in when !do_accept, out otherwise
  int32_t* accept_len;  // in when !do_accept, out otherwise
  int32_t* out_tokens;
  int32_t* bonus;
  // compaction
  int32_t row_bytes, page_size, max_pages;
  int64_t kv_rows;
  uint8_t* kv;
  const int32_t* block_table;
  const int32_t* prefix_len;
  int32_t* new_len;
  int32_t* status;
};
cudaError_t launch_accept_compact(const AcceptCompactArgs& a, cudaStream_t stream);

// B. verify attention, fp32 SIMT path (no workspace).
cudaError_t launch_verify_attn_f32(const ddt_attn_dims& d, const float* q_lat, const float* q_pe,
                                   const float* kv, const int32_t* block_table,
                                   const int32_t* prefix_len, const uint64_t* vis_bits, float* out,
                                   float* lse, int32_t* status, cudaStream_t stream);

// A inside B: the draft tree of each sequence is built by a spare warp of the
// bf16 verify-attention kernel while the prefix part of the attention runs
// (the key tiles that hold tree keys come last in every walk). One cluster
// per sequence writes the tree outputs and OR-s the build's status bits.
struct TreeFuse {
  int32_t D, K, budget, V;
  const float* topk_logp;
  const int32_t* topk_ids;
  const int32_t* root_tok;
  int32_t* tokens;
  int32_t* parents;
  int32_t* depths;
  uint64_t* vis_bits;
  uint8_t* vis;  // may be null
  int32_t* first_child;
  int32_t* next_sibling;
  int32_t* n_nodes;
};
// Largest candidate table (min(D,budget) x min(K,budget)) the fused build stages.
constexpr int kFuseMaxCand = 1024;

// ---- debug-build bounds checks ------------------------------------------------
// With -DDDT_CHECKS, DDT_GUARD(cond, site, status) is false when cond fails,
// after counting the failure in the file's device counters (count, first
// failing site) and OR-ing DDT_ST_CHECK into *status (status may be null).
// Without the flag it is the constant true and cond is not evaluated. Each
// .cu file that uses it names its counters once with DDT_CHECKS_FILE(name);
// checks_read_<name>() reads and resets them (host, synchronising).
#ifdef DDT_CHECKS
__device__ __forceinline__ bool ddt_check_failed(int* chk, int site, int32_t* status) {
  if (atomicAdd(&chk[0], 1) == 0) chk[1] = site;
  if (status != nullptr) atomicOr(status, DDT_ST_CHECK);
  return false;
}
#define DDT_GUARD(cond, site, status) ((cond) ? true : ::ddt::ddt_check_failed(g_chk, (site), (status)))
#define DDT_CHECKS_FILE(name)                                            \
  static __device__ int g_chk[2];                                        \
  int checks_read_##name(int* first) {                                   \
    int h[2] = {0, 0};                                                   \
    const int z[2] = {0, 0};                                             \
    if (cudaMemcpyFromSymbol(h, g_chk, sizeof(h)) != cudaSuccess) h[0] = -1; \
    cudaMemcpyToSymbol(g_chk, z, sizeof(z));                             \
    *first = h[1];                                                       \
    return h[0];                                                         \
  }
#else
#define DDT_GUARD(cond, site, status) true
#define DDT_CHECKS_FILE(name)        \
  int checks_read_##name(int* first) { \
    *first = 0;                      \
    return 0;                        \
  }
#endif
int checks_read_pair(int* first);
int checks_read_bf16(int* first);
int checks_read_f32(int* first);
int checks_read_build(int* first);
int checks_read_accept(int* first);
int checks_read_rope(int* first);
int checks_read_topk(int* first);
int checks_read_argmax(int* first);

// B. verify attention, bf16 tcgen05 path. With `fuse`, vis_bits is not read:
// the kernel builds the tree itself and status must be zero on entry.
size_t verify_attn_bf16_workspace(const ddt_attn_dims& d);
cudaError_t launch_verify_attn_bf16(const ddt_attn_dims& d, const void* q_lat, const void* q_pe,
                                    const void* kv, const int32_t* block_table,
                                    const int32_t* prefix_len, const uint64_t* vis_bits,
                                    void* out, float* lse, int32_t* status, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream,
                                    const TreeFuse* fuse = nullptr,
                                    const AcceptCompactArgs* then = nullptr);

// The 256-row form of the bf16 verify attention (verify_attn_pair.cu): four-CTA
// clusters, MMAs on paired SMs. `part_o` (bf16) / `part_lse` hold the split-KV
// partials when n_split > 1 (merged by the caller).
int verify_attn_pair_clusters_per_wave();
cudaError_t launch_verify_attn_pair(const ddt_attn_dims& d, int n_split, const void* q_lat,
                                    const void* q_pe, const void* kv, const int32_t* block_table,
                                    const int32_t* prefix_len, const uint64_t* vis_bits, void* out,
                                    float* lse, int32_t* status, __nv_bfloat16* part_o,
                                    float* part_lse, cudaStream_t stream, const TreeFuse* fuse);
// Row-tile height (128 or 256) and key-range split the next bf16 launch with
// these dims uses.
int verify_attn_bf16_rows_per_tile(const ddt_attn_dims& d);
int verify_attn_bf16_splits(const ddt_attn_dims& d);

// Target-side argmax over the vocabulary, one row per tree slot.
cudaError_t launch_target_argmax(long long rows, long long V, int dtype, const void* logits,
                                 int32_t* argmax, cudaStream_t stream);

// Drafter-side log-softmax top-K over the vocabulary, one row per (sequence, depth).
cudaError_t launch_drafter_topk(long long rows, long long V, int K, int dtype, const void* logits,
                                float* topk_logp, int32_t* topk_ids, cudaStream_t stream);

// Host checks of a verify-attention call (defined in ddt_api.cu).
int check_verify_attn_args(const ddt_attn_dims* d, const void* q_lat, const void* q_pe,
                           const void* kv, const int32_t* block_table, const int32_t* prefix_len,
                           const uint64_t* vis_bits, const void* out, const int32_t* status);

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device
// (later calls, including ones made while a stream is being captured into a
// CUDA graph, issue no driver call). `done` is the caller's per-kernel cache.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel k, int bytes, int (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = bytes;
  return e;
}

// CTAs per row for the row-streaming kernels (argmax, top-K): the smallest
// power of two up to `max_csize` that puts at least one CTA on every SM.
// Splitting further only adds per-CTA merges; fewer leaves SMs idle.
int device_sm_count();
inline unsigned row_cluster_size(long long rows, int max_csize) {
  const long long want = device_sm_count();
  unsigned c = 1;
  while ((long long)c * rows < want && (int)(2 * c) <= max_csize) c *= 2;
  return c;
}
// Rotary frequencies theta^(-2i/R), i < R/2, computed on the host in double
// and passed by value to the rope kernel.
constexpr int kMaxRopeHalf = 128;
struct RopeFreqs {
  double f[kMaxRopeHalf];
};
cudaError_t launch_rope_append(const ddt_attn_dims& d, const RopeFreqs& freqs,
                               const int32_t* depths, const int32_t* prefix_len,
                               const int32_t* block_table, const void* q_in, void* q_out,
                               const void* kv_new, void* kv, int32_t* status, cudaStream_t stream);

// Launch `kernel` over `grid` CTAs in clusters of `csize` (1: no cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_rows(void (*kernel)(KArgs...), unsigned grid, unsigned csize, unsigned threads,
                        cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = csize;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
// Launch a row-streaming kernel over `rows` rows, each row on a cluster of
// row_cluster_size() CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_row_kernel(void (*kernel)(KArgs...), long long rows, int max_csize,
                              unsigned threads, cudaStream_t stream, Args... args) {
  const unsigned csize = row_cluster_size(rows, max_csize);
  if (rows < 1 || rows * csize > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_rows(kernel, (unsigned)(rows * csize), csize, threads, stream, args...);
}

// ---- small device helpers ----------------------------------------------------

__device__ __forceinline__ int64_t slot_row(const int32_t* __restrict__ bt_row, int32_t page_size,
                                            int64_t slot) {
  const int64_t page = bt_row[slot / page_size];
  return page * page_size + slot % page_size;
}

__device__ __forceinline__ bool warp_any(bool p) { return __any_sync(0xffffffffu, p); }

}  // namespace ddt
