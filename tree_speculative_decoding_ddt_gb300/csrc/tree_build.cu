// A. Best-first draft-tree construction on the GPU: one warp per sequence,
// several sequences per CTA.
// The algorithm and its GB300 layout are described in tree_build_warp.cuh;
// this kernel runs it for every sequence of the batch and writes the tree.
#include "tree_build_warp.cuh"

namespace ddt {
DDT_CHECKS_FILE(build)
namespace {

constexpr int kWarpsPerCta = 4;  // sequences per CTA, one warp each

template <int NS>
__global__ void __launch_bounds__(32 * kWarpsPerCta) k_tree_build(
    int B, int D, int K, int budget, int V, int De, int Ke, int warp_smem,
    const float* __restrict__ topk_logp, const int32_t* __restrict__ topk_ids,
    const int32_t* __restrict__ root_tok, int32_t* __restrict__ tokens,
    int32_t* __restrict__ parents, int32_t* __restrict__ depths,
    unsigned long long* __restrict__ vis_bits, uint8_t* __restrict__ vis,
    int32_t* __restrict__ first_child, int32_t* __restrict__ next_sibling,
    int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= B) return;  // warps are independent: no CTA-wide barrier below
  unsigned char* mine = smem_raw + (size_t)warp * warp_smem;
  tb::Smem& S = *reinterpret_cast<tb::Smem*>(mine);
  double* s_logp = reinterpret_cast<double*>(mine + sizeof(tb::Smem));  // [De][Ke]
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_logp + De * Ke);       // [De][Ke]
  bool bad = false;
  const int n = tb::build_warp<NS>(topk_logp + (size_t)b * D * K, topk_ids + (size_t)b * D * K,
                                   root_tok[b], D, K, budget, V, De, Ke, S, s_logp, s_ids, &bad);
  const int32_t st = tb::write_warp(S, b, budget + 1, n, bad, tokens, parents, depths, vis_bits,
                                    vis, first_child, next_sibling, n_nodes_out);
  if ((threadIdx.x & 31) == 0) status[b] = st;
  // the pop loop yields the root and at most `budget` nodes
  if ((threadIdx.x & 31) == 0) (void)DDT_GUARD(n >= 1 && n <= budget + 1, 401, status + b);
}

}  // namespace

cudaError_t launch_tree_build(const ddt_tree_dims& d, const float* topk_logp,
                              const int32_t* topk_ids, const int32_t* root_tok, int32_t* tokens,
                              int32_t* parents, int32_t* depths, uint64_t* vis_bits, uint8_t* vis,
                              int32_t* first_child, int32_t* next_sibling, int32_t* n_nodes,
                              int32_t* status, cudaStream_t stream) {
  const int De = d.D < d.budget ? d.D : d.budget;
  const int Ke = d.K < d.budget ? d.K : d.budget;
  // one warp per sequence, kWarpsPerCta sequences per CTA (fewer warps when
  // the batch is smaller), each warp with its own shared-memory area
  const int warp_smem = (int)((tb::smem_bytes(De, Ke) + 15) & ~size_t(15));
  int wpc = d.B < kWarpsPerCta ? d.B : kWarpsPerCta;
  while (wpc > 1 && (size_t)warp_smem * wpc > 200 * 1024) --wpc;  // large candidate tables
  const size_t smem = (size_t)warp_smem * wpc;
  const int ns = tb::slots_for(d.budget + 1);
  auto kern = ns == 1 ? k_tree_build<1> : ns == 2 ? k_tree_build<2> : ns == 3 ? k_tree_build<3>
                                                                             : k_tree_build<4>;
  static int smem_set[4][64] = {};
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit(kern, (int)smem, smem_set[ns - 1]);
    if (e != cudaSuccess) return e;
  }
  const int grid = (d.B + wpc - 1) / wpc;
  kern<<<grid, 32 * wpc, smem, stream>>>(d.B, d.D, d.K, d.budget, d.V, De, Ke, warp_smem,
                                         topk_logp, topk_ids, root_tok, tokens, parents, depths,
                                         reinterpret_cast<unsigned long long*>(vis_bits), vis,
                                         first_child, next_sibling, n_nodes, status);
  return cudaGetLastError();
}

}  // namespace ddt
