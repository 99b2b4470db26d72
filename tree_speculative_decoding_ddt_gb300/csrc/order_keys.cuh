// 64-bit ranking keys of vocabulary entries, shared by the kernels that pick
// the largest logits (target argmax, drafter top-K): the upper 32 bits are an
// order-preserving image of the value, the lower 32 bits the complemented
// column, so a larger key is a larger value, and among equal values the
// lower column.
#pragma once

#include <stdint.h>

namespace ddt {
namespace keys {

// A larger value maps to a larger image; -0.0 and +0.0 map to the same image;
// every NaN maps above +inf.
__device__ __forceinline__ uint32_t order_of(uint16_t h) {  // bf16 bits
  if ((h & 0x7F80u) == 0x7F80u && (h & 0x007Fu)) return 0xFFFFFFFFu;
  if (h == 0x8000u) h = 0;
  return (h & 0x8000u) ? (uint32_t)(~h & 0xFFFFu) : (uint32_t)(h | 0x8000u);
}
__device__ __forceinline__ uint32_t order_of(uint32_t u) {  // f32 bits
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0xFFFFFFFFu;
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// the value back from a non-NaN image (+0.0 for either zero)
__device__ __forceinline__ float value_of_bf16(uint32_t ord) {
  const uint32_t h = (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
  return __uint_as_float(h << 16);
}
__device__ __forceinline__ float value_of_f32(uint32_t ord) {
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

__device__ __forceinline__ unsigned long long key_of(uint32_t ord, uint32_t col) {
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - col);
}
__device__ __forceinline__ uint32_t col_of(unsigned long long key) {
  return 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
}
__device__ __forceinline__ unsigned long long max_key(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// CTAs in this CTA's cluster (1 for a launch without clusters) and its rank.
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

}  // namespace keys
}  // namespace ddt
