// Drafter-side log-softmax and per-depth top-K over the vocabulary.
//
// "The Milestone Commit: Cementing a Native DDTree Inference Engine", section
// "What the Message Actually Does": the GPU tree builder consumes the
// drafter's per-depth top-K log-probabilities; the verify-step specification
// scores a node by the sum of the log-probs along its path. This is the step
// just upstream of the build: rows = (sequence, depth), columns = the
// vocabulary; per row the K largest logits (value descending, token id
// ascending on ties) and logit - log(sum(exp(logits))).
//
// HBM-bound: every logit is read once. Each row is read by a cluster of 1 to 8
// CTAs (as few as still put a CTA on every SM), each CTA streaming its share
// of the row with 16-byte loads. A thread keeps an online log-sum-exp (running
// max, rescaled sum, one exp2 per logit) and a descending list of K ranking
// keys (order_keys.cuh; K rounded up to a power of two), touched only when a
// vector's maximum reaches both the list's last key and a lower bound on the
// row's K-th value: first the K-th largest of the lanes' first maxima, then
// the warp's K-th best, shared across the CTA through one shared-memory
// maximum. Lists merge by K rounds of "the largest head wins and its list
// advances": within a warp, across the CTA's warps, then across the cluster's
// CTAs through distributed shared memory, where the rank-0 CTA also combines
// the (max, sum) pairs.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"
#include "order_keys.cuh"
#include "sm100_ptx.cuh"

namespace ddt {
DDT_CHECKS_FILE(topk)
namespace {

using namespace sm100;
using keys::key_of;
using keys::order_of;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxK = 16;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A running (max m, sum s of exp(x - m)) of a set of logits; -inf / 0 = empty.
struct Lse {
  float m = -INFINITY;
  float s = 0.f;
  __device__ void add(const Lse& o) {
    if (o.m == -INFINITY) return;
    if (m == -INFINITY) {
      *this = o;
      return;
    }
    const float M = fmaxf(m, o.m);
    s = s * ex2f((m - M) * kLog2e) + o.s * ex2f((o.m - M) * kLog2e);
    m = M;
  }
};

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
  __device__ static uint32_t ord(float x) { return order_of((uint16_t)(__float_as_uint(x) >> 16)); }
  __device__ static float value(uint32_t o) { return keys::value_of_bf16(o); }
  __device__ static float pick(const float (&f)[8], int j) {  // f[j] by selects
    const float a0 = (j & 1) ? f[1] : f[0], a1 = (j & 1) ? f[3] : f[2];
    const float a2 = (j & 1) ? f[5] : f[4], a3 = (j & 1) ? f[7] : f[6];
    const float b0 = (j & 2) ? a1 : a0, b1 = (j & 2) ? a3 : a2;
    return (j & 4) ? b1 : b0;
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
  __device__ static uint32_t ord(float x) { return order_of(__float_as_uint(x)); }
  __device__ static float value(uint32_t o) { return keys::value_of_f32(o); }
  __device__ static float pick(const float (&f)[4], int j) {  // f[j] by selects
    const float a0 = (j & 1) ? f[1] : f[0], a1 = (j & 1) ? f[3] : f[2];
    return (j & 2) ? a1 : a0;
  }
  __device__ static float scalar(const float* p) { return *p; }
};

// The KT best (value, column) pairs one thread has seen, in rank order
// (value descending, then column ascending); empty slots hold (-inf, none).
// KT is K rounded up to a power of two, a compile-time length so that every
// index is a constant and the list stays in registers. The filter is one
// float compare per logit against the last value; the exact rank comparison
// runs only for logits that reach it.
constexpr uint32_t kNone = 0xFFFFFFFFu;
template <int KT>
struct TopList {
  float v[KT];
  uint32_t c[KT];
  __device__ void clear() {
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      v[j] = -INFINITY;
      c[j] = kNone;
    }
  }
  __device__ float last() const { return v[KT - 1]; }
  __device__ static bool ahead(float f, uint32_t col, float vj, uint32_t cj) {
    return f > vj || (f == vj && col < cj);
  }
  // insert (f, col) at its rank, dropping the last entry
  __device__ void insert(float f, uint32_t col) {
#pragma unroll
    for (int j = KT - 1; j >= 0; --j) {
      if (!ahead(f, col, v[j], c[j])) continue;
      if (j > 0 && ahead(f, col, v[j - 1], c[j - 1])) {
        v[j] = v[j - 1];
        c[j] = c[j - 1];
      } else {
        v[j] = f;
        c[j] = col;
      }
    }
  }
};

// Descending 64-bit ranking keys (order_keys.cuh) for the merges.
template <int KT>
struct TopK {
  unsigned long long k[KT];
  __device__ void clear() {
#pragma unroll
    for (int j = 0; j < KT; ++j) k[j] = 0ull;
  }
  // drop the head (it won a merge round)
  __device__ void pop() {
#pragma unroll
    for (int j = 0; j < KT - 1; ++j) k[j] = k[j + 1];
    k[KT - 1] = 0ull;
  }
};

__device__ __forceinline__ unsigned long long warp_max(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}
// K rounds over the lanes' lists: round r appends the largest head to out[r]
// (lane 0 writes) and pops it from the lane that held it (keys are unique:
// the column is part of the key).
template <int KT>
__device__ void warp_merge(TopK<KT>& t, int K, unsigned long long* out) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < K; ++r) {
    const unsigned long long w = warp_max(t.k[0]);
    if (lane == 0) out[r] = w;
    if (w != 0ull && t.k[0] == w) t.pop();
  }
}
// The K-th largest value over the lists of all lanes of the warp (-inf if
// the warp has seen fewer than K logits). No logit below it can be in the
// row's top K, so it is a safe filter for every lane. Values alone suffice
// for a bound: K rounds of "the warp maximum of the heads, the lowest lane
// holding it advances".
template <int KT>
__device__ float warp_kth(const TopList<KT>& tl, int K) {
  float h[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) h[j] = tl.v[j];
  const int lane = threadIdx.x & 31;
  float w = -INFINITY;
  for (int r = 0; r < K; ++r) {
    w = h[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, off));
    const unsigned holders = __ballot_sync(0xffffffffu, h[0] == w);
    if (lane == __ffs(holders) - 1) {
#pragma unroll
      for (int j = 0; j < KT - 1; ++j) h[j] = h[j + 1];
      h[KT - 1] = -INFINITY;
    }
  }
  return w;
}

// The K-th largest of the lanes' values x (-inf if fewer than K lanes hold a
// number): K rounds of "take the warp maximum, the lowest lane holding it
// drops out".
__device__ float warp_kth_value(float x, int K) {
  const int lane = threadIdx.x & 31;
  float w = -INFINITY;
  for (int r = 0; r < K; ++r) {
    w = x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, off));
    const unsigned holders = __ballot_sync(0xffffffffu, x == w);
    if (lane == __ffs(holders) - 1) x = -INFINITY;
  }
  return w;
}

__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// kIF: 16-byte loads a thread issues before using any. Three launch shapes:
// rows that fill more than three CTAs per SM take 6 loads in flight and at
// most 64 registers (K <= 8), so four CTAs fit per SM and the grid runs as
// one wave; small shares (up to 32 vectors a thread) take 16 with two CTAs
// per SM, so one or two batches cover them and a cluster of eight still
// finds room; the rest take 8 with three CTAs per SM.
template <typename T, int KT, int kIF, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    k_drafter_topk(const T* __restrict__ logits, long long V, int K, int vec,
                   float* __restrict__ topk_logp, int32_t* __restrict__ topk_ids) {
  using E = Elems<T>;
  __shared__ unsigned long long s_warp[kWarps][kMaxK];
  __shared__ float s_wm[kWarps], s_ws[kWarps];
  __shared__ unsigned long long s_cta[kMaxK];
  __shared__ float s_cm, s_cs;
  // the best lower bound on the row's K-th value that a warp of this CTA has
  // found, as an order image of its f32 bits (order_keys.cuh)
  __shared__ uint32_t s_thr;
  const uint32_t ncta = keys::cluster_size();  // the row's CTAs
  const long long row = blockIdx.x / ncta;
  const uint32_t crank = cluster_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* x = logits + row * V;

  const long long per = (((V + ncta - 1) / ncta) + E::kPerVec - 1) / E::kPerVec * E::kPerVec;
  const long long c0 = min(V, (long long)crank * per);
  const long long c1 = min(V, c0 + per);
  if (tid == 0) (void)DDT_GUARD(c0 >= 0 && c0 <= c1 && c1 <= V, 701, nullptr);
  TopList<KT> tl;
  tl.clear();
  Lse ls;
  float wthr = -INFINITY;  // a lower bound on the row's K-th value (the filter)
  if (tid == 0) s_thr = order_of(__float_as_uint(-INFINITY));
  __syncthreads();
  if (vec) {
    const long long nv = (c1 - c0) / E::kPerVec;
    const uint4* xv = reinterpret_cast<const uint4*>(x + c0);
    for (long long base = 0; base < nv; base += (long long)kThreads * kIF) {
      uint4 v[kIF];
#pragma unroll
      for (int k = 0; k < kIF; ++k) {
        const long long i = base + tid + (long long)k * kThreads;
        if (i < nv) v[k] = ld_stream(xv + i);
      }
      if (base == 0) {
        // before any list exists: the maxima of the lanes' first vectors
        // are distinct logits, so the K-th largest of them bounds the row's
        // K-th value from below and spares the lanes most first inserts
        float lm = -INFINITY;
#pragma unroll
        for (int k = 0; k < kIF; ++k) {
          if (base + tid + (long long)k * kThreads >= nv) continue;
          float f[E::kPerVec];
          E::unpack(v[k], f);
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) lm = fmaxf(lm, f[j]);
        }
        wthr = warp_kth_value(lm, K);
      }
#pragma unroll
      for (int k = 0; k < kIF; ++k) {
        const long long i = base + tid + (long long)k * kThreads;
        if (i >= nv) continue;
        float f[E::kPerVec];
        E::unpack(v[k], f);
        float vm = f[0];
#pragma unroll
        for (int j = 1; j < E::kPerVec; ++j) vm = fmaxf(vm, f[j]);
        if (vm > ls.m) {
          if (ls.m != -INFINITY) ls.s *= ex2f((ls.m - vm) * kLog2e);
          ls.m = vm;
        }
        if (ls.m != -INFINITY) {
          const float nm = -ls.m * kLog2e;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) acc += ex2f(fmaf(f[j], kLog2e, nm));
          ls.s += acc;
        }
        // the list changes only if the vector reaches both the list's last
        // value and the lower bound on the row's K-th value (ties still go
        // through: the column decides them)
        if (vm >= fmaxf(tl.last(), wthr)) {
          const uint32_t col0 = (uint32_t)(c0 + i * E::kPerVec);
          // visit only the elements that reach the filter (usually one),
          // in column order, picking each by a select tree (no indexing)
          const float thr = fmaxf(tl.last(), wthr);
          uint32_t mask = 0;
#pragma unroll
          for (int j = 0; j < E::kPerVec; ++j) mask |= (f[j] >= thr ? 1u : 0u) << j;
          while (mask) {
            const int j = __ffs(mask) - 1;
            mask &= mask - 1;
            const float fj = E::pick(f, j);
            if (fj >= fmaxf(tl.last(), wthr)) tl.insert(fj, col0 + (uint32_t)j);
          }
        }
      }
      // a lane alone sees few logits, so its own K-th best stays low and some
      // lane of the warp would take the insert path at nearly every vector:
      // tighten every lane's filter to the warp's K-th best
      wthr = fmaxf(wthr, warp_kth(tl, K));
      // and share the bound with the CTA's other warps
      if (lane == 0) atomicMax(&s_thr, order_of(__float_as_uint(wthr)));
      __syncwarp();
      wthr = fmaxf(wthr, keys::value_of_f32(*static_cast<volatile uint32_t*>(&s_thr)));
    }
  } else {
    for (long long c = c0 + tid; c < c1; c += kThreads) {
      const float f = E::scalar(x + c);
      Lse one;
      one.m = f;
      one.s = f == -INFINITY ? 0.f : 1.f;
      ls.add(one);
      if (f >= tl.last()) tl.insert(f, (uint32_t)c);
    }
  }
  TopK<KT> tk;
#pragma unroll
  for (int j = 0; j < KT; ++j)
    tk.k[j] = tl.c[j] == kNone ? 0ull : key_of(E::ord(tl.v[j]), tl.c[j]);

  // ---- warp, CTA, cluster merges of the lists and of the (max, sum) pairs
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Lse o;
    o.m = __shfl_xor_sync(0xffffffffu, ls.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, ls.s, off);
    ls.add(o);
  }
  warp_merge(tk, K, s_warp[warp]);
  if (lane == 0) {
    s_wm[warp] = ls.m;
    s_ws[warp] = ls.s;
  }
  __syncthreads();
  if (warp == 0) {
    tk.clear();
    if (lane < kWarps)
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (j < K) tk.k[j] = s_warp[lane][j];
    warp_merge(tk, K, s_cta);
    if (lane == 0) {
      Lse c;
      for (int w = 0; w < kWarps; ++w) {
        Lse o;
        o.m = s_wm[w];
        o.s = s_ws[w];
        c.add(o);
      }
      s_cm = c.m;
      s_cs = c.s;
    }
  }
  cluster_sync();  // every CTA's list and pair are in its shared memory
  if (crank == 0 && warp == 0) {
    __shared__ unsigned long long s_out[kMaxK];
    tk.clear();
    if (lane < (int)ncta) {
      const uint32_t base = map_peer(smem_u32(s_cta), (uint32_t)lane);
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (j < K) tk.k[j] = ld_cluster_u64(base + 8u * j);
    }
    warp_merge(tk, K, s_out);
    Lse c;
    if (lane < (int)ncta) {
      c.m = ld_cluster_f32(map_peer(smem_u32(&s_cm), (uint32_t)lane));
      c.s = ld_cluster_f32(map_peer(smem_u32(&s_cs), (uint32_t)lane));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      Lse o;
      o.m = __shfl_xor_sync(0xffffffffu, c.m, off);
      o.s = __shfl_xor_sync(0xffffffffu, c.s, off);
      c.add(o);
    }
    __syncwarp();
    const float lse = c.m + logf(c.s);
    if (lane < K) {
      const unsigned long long key = s_out[lane];
      topk_logp[row * K + lane] = E::value((uint32_t)(key >> 32)) - lse;
      topk_ids[row * K + lane] = (int32_t)keys::col_of(key);
    }
  }
  cluster_sync();  // the peers' shared memory stays valid until rank 0 has read it
}

}  // namespace

cudaError_t launch_drafter_topk(long long rows, long long V, int K, int dtype, const void* logits,
                                float* topk_logp, int32_t* topk_ids, cudaStream_t stream) {
  if (rows < 1 || V < 1 || K < 1 || K > kMaxK || K > V) return cudaErrorInvalidValue;
  const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  const int vb = aligned && V % 8 == 0, vf = aligned && V % 4 == 0;
  const __nv_bfloat16* lb = static_cast<const __nv_bfloat16*>(logits);
  const float* lf = static_cast<const float*>(logits);
  // the launch shape (see k_drafter_topk)
  const int sms = device_sm_count();
  const unsigned csize = row_cluster_size(rows, kMaxCluster);
  const long long per_thread =
      ((V + csize - 1) / csize + 8LL * kThreads - 1) / (8LL * kThreads);  // bf16 vectors
  const int shape = rows * csize > 3LL * sms ? 0 : (per_thread <= 32 ? 1 : 2);
#define DDT_TOPK_SHAPE(KT, IF, MB)                                                            \
  return dtype == DDT_BF16                                                                    \
             ? launch_row_kernel(k_drafter_topk<__nv_bfloat16, KT, IF, MB>, rows, kMaxCluster, \
                                 kThreads, stream, lb, V, K, vb, topk_logp, topk_ids)         \
             : launch_row_kernel(k_drafter_topk<float, KT, IF, MB>, rows, kMaxCluster,         \
                                 kThreads, stream, lf, V, K, vf, topk_logp, topk_ids);
#define DDT_TOPK_LAUNCH(KT)                 \
  {                                         \
    if (shape == 0) DDT_TOPK_SHAPE(KT, 6, (KT >= 16 ? 2 : 4)) \
    if (shape == 1) DDT_TOPK_SHAPE(KT, 16, 2) \
    DDT_TOPK_SHAPE(KT, 8, (KT >= 16 ? 2 : 3)) \
  }
  if (K <= 1) DDT_TOPK_LAUNCH(1)
  if (K <= 2) DDT_TOPK_LAUNCH(2)
  if (K <= 4) DDT_TOPK_LAUNCH(4)
  if (K <= 8) DDT_TOPK_LAUNCH(8)
  DDT_TOPK_LAUNCH(16)
#undef DDT_TOPK_SHAPE
#undef DDT_TOPK_LAUNCH
}

}  // namespace ddt
