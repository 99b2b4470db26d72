// Target-side argmax over the vocabulary at every tree slot.
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": the target model's greedy token at each tree node (the argmax of
// its logits) is what tree_accept compares the drafted tokens with. This is
// the step just upstream of accept: rows = tree slots of all sequences,
// columns = the vocabulary.
//
// HBM-bound: every logit is read once. Each row is read by a cluster of 1 to 8
// CTAs (as few as still put a CTA on every SM); each CTA streams its share of
// the row with 16-byte loads (eight in flight per thread). A thread scans its
// vectors in column order with about two instructions per logit (widen, NaN-
// propagating max per vector) and looks for a column only when a vector beats
// its running best. The thread results meet as 64-bit keys -- order-preserving
// value bits above the complemented column, so the largest key is the largest
// value at the lowest column -- in warp, CTA and finally the rank-0 CTA of the
// cluster through distributed shared memory. One launch, no scratch memory.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ddt_internal.cuh"
#include "order_keys.cuh"
#include "sm100_ptx.cuh"

namespace ddt {
DDT_CHECKS_FILE(argmax)
namespace {

using namespace sm100;

constexpr int kThreads = 256;
constexpr int kMaxCluster = 8;
constexpr int kInFlight = 8;  // 16-byte loads issued before any is used

using keys::key_of;
using keys::max_key;
using keys::order_of;

__device__ __forceinline__ float max_nan(float a, float b) {  // NaN if either is NaN
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The elements of one 16-byte vector as floats (exact), in column order.
template <typename T>
struct Elems;
template <>
struct Elems<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static void unpack(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static uint32_t order_bits(float x) {
    return order_of((uint16_t)(__float_as_uint(x) >> 16));
  }
  __device__ static float scalar(const __nv_bfloat16* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
};
template <>
struct Elems<float> {
  static constexpr int kPerVec = 4;
  __device__ static void unpack(uint4 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint32_t order_bits(float x) { return order_of(__float_as_uint(x)); }
  __device__ static float scalar(const float* p) { return *p; }
};

// Running best of one thread, fed in increasing column order: replaced only
// by a strictly larger value (or the first NaN), so among equal values (and
// -0.0 == +0.0) the earliest column stays.
struct Best {
  float v = 0.f;
  long long col = -1;  // none yet
  __device__ bool beaten_by(float x) const {
    return col < 0 || (x > v) || (x != x && v == v);
  }
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

// vec: every row starts on a 16-byte boundary and V is a multiple of the
// elements per 16 bytes, so the whole row is read with vector loads
template <typename T>
__global__ void __launch_bounds__(kThreads)
    k_target_argmax(const T* __restrict__ logits, long long V, int vec, int32_t* __restrict__ out) {
  using E = Elems<T>;
  __shared__ unsigned long long s_warp[kThreads / 32];
  __shared__ unsigned long long s_cta;
  const uint32_t ncta = keys::cluster_size();  // the row's CTAs
  const long long row = blockIdx.x / ncta;
  const uint32_t crank = cluster_rank();
  const int tid = threadIdx.x;
  const T* x = logits + row * V;

  // this CTA's columns [c0, c1): an eighth of the row, in whole vectors
  const long long per = (((V + ncta - 1) / ncta) + E::kPerVec - 1) / E::kPerVec * E::kPerVec;
  const long long c0 = min(V, (long long)crank * per);
  const long long c1 = min(V, c0 + per);
  if (tid == 0) (void)DDT_GUARD(c0 >= 0 && c0 <= c1 && c1 <= V, 801, nullptr);
  Best bt;
  if (vec) {
    const long long nv = (c1 - c0) / E::kPerVec;
    const uint4* xv = reinterpret_cast<const uint4*>(x + c0);
    for (long long base = 0; base < nv; base += (long long)kThreads * kInFlight) {
      uint4 v[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const long long i = base + tid + (long long)k * kThreads;
        if (i < nv) v[k] = ld_stream(xv + i);
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const long long i = base + tid + (long long)k * kThreads;
        if (i >= nv) continue;
        float f[E::kPerVec];
        E::unpack(v[k], f);
        float m = f[0];
#pragma unroll
        for (int j = 1; j < E::kPerVec; ++j) m = max_nan(m, f[j]);
        if (bt.beaten_by(m)) {  // rare after the first vectors: find m's first column
          int jf = 0;
#pragma unroll
          for (int j = E::kPerVec - 1; j >= 0; --j)
            if (f[j] == m || (m != m && f[j] != f[j])) jf = j;
          bt.v = m;
          bt.col = c0 + i * E::kPerVec + jf;
        }
      }
    }
  } else {
    for (long long c = c0 + tid; c < c1; c += kThreads) {
      const float xv = E::scalar(x + c);
      if (bt.beaten_by(xv)) {
        bt.v = xv;
        bt.col = c;
      }
    }
  }
  unsigned long long best =
      bt.col < 0 ? 0ull : key_of(E::order_bits(bt.v), (uint32_t)bt.col);
  // warp, CTA, then cluster maximum
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    best = max_key(best, __shfl_xor_sync(0xffffffffu, best, off));
  if ((tid & 31) == 0) s_warp[tid >> 5] = best;
  __syncthreads();
  if (tid == 0) {
    unsigned long long b = s_warp[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) b = max_key(b, s_warp[w]);
    s_cta = b;
  }
  cluster_sync();  // every CTA's result is in its shared memory
  if (crank == 0 && tid == 0) {
    unsigned long long b = s_cta;
    const uint32_t local = smem_u32(&s_cta);
    for (uint32_t r = 1; r < ncta; ++r) b = max_key(b, ld_cluster_u64(map_peer(local, r)));
    out[row] = (int32_t)keys::col_of(b);
  }
  cluster_sync();  // the peers' shared memory stays valid until rank 0 has read it
}

}  // namespace

cudaError_t launch_target_argmax(long long rows, long long V, int dtype, const void* logits,
                                 int32_t* argmax, cudaStream_t stream) {
  if (rows < 1 || V < 1) return cudaErrorInvalidValue;
  const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  if (dtype == DDT_BF16)
    return launch_row_kernel(k_target_argmax<__nv_bfloat16>, rows, kMaxCluster, kThreads, stream,
                             static_cast<const __nv_bfloat16*>(logits), V,
                             (int)(aligned && V % 8 == 0), argmax);
  return launch_row_kernel(k_target_argmax<float>, rows, kMaxCluster, kThreads, stream,
                           static_cast<const float*>(logits), V, (int)(aligned && V % 4 == 0),
                           argmax);
}

}  // namespace ddt
