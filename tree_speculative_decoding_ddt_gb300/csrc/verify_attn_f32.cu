// B. Tree-verify MLA-absorb attention, fp32 exactness path (SIMT).
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": attention runs through a custom verify_attn kernel in MLA absorb
// form over the latent cache; the tree [verified_id, drafts] sits at cache
// positions L + depth and the mask is [ones over the prefix | visibility].
// The engine on those pages runs in FP32 throughout ("Assumptions Made"), so
// this path keeps every product and sum in fp32 for parity checks at any
// C/R (the odd dims of the second validation model included).
//
// One CTA per (sequence, tree query, group of 8 heads); one warp per head.
// A tile of 32 cache rows is staged in shared memory once and reused by the
// 8 heads; the row stride is padded by one float so that lane j reading
// row j is bank-conflict free. Online softmax in natural-log units.
#include <math.h>

#include "ddt_internal.cuh"

namespace ddt {
DDT_CHECKS_FILE(f32)
namespace {

constexpr int kHeads = 8;
constexpr int kTile = 32;
constexpr int kMaxCPerLane = 32;  // C <= 1024

__global__ void __launch_bounds__(kHeads * 32) k_verify_attn_f32(
    int B, int Q, int H, int C, int R, int page_size, int max_pages, long long kv_rows, float scale,
    const float* __restrict__ q_lat, const float* __restrict__ q_pe, const float* __restrict__ kv,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ prefix_len,
    const unsigned long long* __restrict__ vis_bits, float* __restrict__ out,
    float* __restrict__ lse_out, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) float sm[];
  const int CR = C + R;
  const int ld = CR + 1;
  float* q_s = sm;                  // [kHeads][CR]
  float* kv_s = sm + kHeads * CR;   // [kTile][CR + 1]

  const int b = blockIdx.x / Q;
  const int i = blockIdx.x % Q;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * kHeads + warp;
  const int W = (Q + 63) / 64;
  const int32_t* bt = block_table + (size_t)b * max_pages;

  // ---- capacity and page checks (the same decision in every CTA of b) -----
  const long long L = prefix_len[b];
  const long long n_keys = L + Q;
  int code = 0;
  if (L < 0 || n_keys > (long long)max_pages * page_size) code = DDT_ST_CAPACITY;
  if (code == 0) {
    const long long n_pages = (n_keys + page_size - 1) / page_size;
    bool badp = false;
    const long long kv_pages = kv_rows / page_size;  // whole pages only
    for (long long p = threadIdx.x; p < n_pages; p += blockDim.x) {
      const long long pg = bt[p];
      if (pg < 0 || pg >= kv_pages) badp = true;
    }
    if (__syncthreads_or(badp)) code = DDT_ST_RANGE;
  }
  if (code != 0) {
    if (h < H) {
      float* o = out + (((size_t)b * Q + i) * H + h) * C;
      for (int d = lane; d < C; d += 32) o[d] = 0.f;
      if (lse_out && lane == 0) lse_out[((size_t)b * Q + i) * H + h] = -INFINITY;
    }
    if (i == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(status + b, code);
    return;
  }

  // ---- stage this CTA's query rows ----------------------------------------
  for (int e = threadIdx.x; e < kHeads * CR; e += blockDim.x) {
    const int hh = blockIdx.y * kHeads + e / CR, d = e % CR;
    float v = 0.f;
    if (hh < H) {
      const size_t row = ((size_t)b * Q + i) * H + hh;
      v = d < C ? q_lat[row * C + d] : q_pe[row * R + (d - C)];
    }
    q_s[e] = v;
  }
  unsigned long long vis_w[kMaxW];
#pragma unroll
  for (int w = 0; w < kMaxW; ++w) vis_w[w] = w < W ? vis_bits[((size_t)b * Q + i) * W + w] : 0ull;

  float o[kMaxCPerLane];
#pragma unroll
  for (int k = 0; k < kMaxCPerLane; ++k) o[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float* qh = q_s + warp * CR;

  for (long long t0 = 0; t0 < n_keys; t0 += kTile) {
    __syncthreads();
    for (int j = warp; j < kTile; j += kHeads) {
      const long long slot = t0 + j;
      float* dst = kv_s + j * ld;
      const long long srow = slot < n_keys ? slot_row(bt, page_size, slot) : 0;
      if (slot < n_keys && DDT_GUARD(srow >= 0 && srow < kv_rows, 301, status + b)) {
        const float* src = kv + srow * CR;
        for (int d = lane; d < CR; d += 32) dst[d] = src[d];
      } else {
        for (int d = lane; d < CR; d += 32) dst[d] = 0.f;
      }
    }
    __syncthreads();

    // score of key t0 + lane
    const long long slot = t0 + lane;
    bool visible = slot < n_keys;
    if (visible && slot >= L) {
      const int t = (int)(slot - L);
      visible = (vis_w[t >> 6] >> (t & 63)) & 1ull;
    }
    float s = -INFINITY;
    if (visible) {
      const float* kr = kv_s + lane * ld;
      float acc = 0.f;
      for (int d = 0; d < CR; ++d) acc = fmaf(qh[d], kr[d], acc);
      s = acc * scale;
    }
    float mt = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float m_new = fmaxf(m, mt);
    if (m_new == -INFINITY) continue;  // nothing visible so far
    const float alpha = expf(m - m_new);
    const float p = expf(s - m_new);
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int k = 0; k < kMaxCPerLane; ++k) o[k] *= alpha;
    for (int j = 0; j < kTile; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const float* kr = kv_s + j * ld;
#pragma unroll
      for (int k = 0; k < kMaxCPerLane; ++k) {
        const int d = lane + 32 * k;
        if (d < C) o[k] = fmaf(pj, kr[d], o[k]);
      }
    }
    m = m_new;
  }

  if (h < H) {
    float* orow = out + (((size_t)b * Q + i) * H + h) * C;
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < kMaxCPerLane; ++k) {
      const int d = lane + 32 * k;
      if (d < C) orow[d] = o[k] * inv;
    }
    if (lse_out && lane == 0) lse_out[((size_t)b * Q + i) * H + h] = m + logf(l);
  }
}

}  // namespace

cudaError_t launch_verify_attn_f32(const ddt_attn_dims& d, const float* q_lat, const float* q_pe,
                                   const float* kv, const int32_t* block_table,
                                   const int32_t* prefix_len, const uint64_t* vis_bits, float* out,
                                   float* lse, int32_t* status, cudaStream_t stream) {
  const int CR = d.C + d.R;
  const size_t smem = sizeof(float) * ((size_t)kHeads * CR + (size_t)kTile * (CR + 1));
  static int smem_set[64] = {};
  cudaError_t e = ensure_smem_limit(k_verify_attn_f32, (int)smem, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(d.B * d.Q), (unsigned)((d.H + kHeads - 1) / kHeads));
  k_verify_attn_f32<<<grid, kHeads * 32, smem, stream>>>(
      d.B, d.Q, d.H, d.C, d.R, d.page_size, d.max_pages, (long long)d.kv_rows, d.scale, q_lat,
      q_pe, kv, block_table, prefix_len, reinterpret_cast<const unsigned long long*>(vis_bits),
      out, lse, status);
  return cudaGetLastError();
}

}  // namespace ddt
