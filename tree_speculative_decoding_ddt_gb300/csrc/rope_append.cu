// Rotary embedding of the tree at positions L+depth and append of the tree
// latents to the paged cache, the step just before the verify attention.
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": the verify forward processes [verified_id, drafts] at positions
// L+depth with prefix = cache length, and the model appends the new latents
// to the cache before attention; "The Consolidation Point: Validating
// Generality and Wrapping the MVP", section "The Journey to This Point": the
// rotary embedding is the NeoX kind (pair i with i + R/2, frequency
// theta^(-2i/R)).
//
// HBM-bound and small: one CTA per tree slot reads the slot's H query rope
// parts and its latent row once and writes them once (q in place or to a
// second buffer, the latent row to cache slot L + t through the page table).
// The loads that need no position are issued first, so they are in flight
// while the length, the pages and the angles are looked up.
// The R/2 angles of a slot are formed in double (position times a frequency
// the host computed in double, then reduced modulo 2*pi), so the float
// sine and cosine see an argument below pi whatever the position; the pairs
// turn in fp32 and are rounded once to the element type. 16-byte vectors
// wherever the rows allow them.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
DDT_CHECKS_FILE(rope)
namespace {

constexpr int kThreads = 128;
constexpr int kPre = 2;  // query chunks per thread loaded ahead
constexpr int kMaxHalf = kMaxRopeHalf;

struct RopeArgs {
  int B, Q, H, C, R, page_size, max_pages;
  long long kv_rows;
  const int32_t* depths;
  const int32_t* prefix_len;
  const int32_t* block_table;
  const void* q_in;
  void* q_out;
  const void* kv_new;
  void* kv;
  int32_t* status;
  int vec;  // rows and halves allow 16-byte vectors
  RopeFreqs freqs;
};

template <typename T>
struct El;
template <>
struct El<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static float get(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }
  __device__ static void put(__nv_bfloat16* p, long long i, float x) { p[i] = __float2bfloat16_rn(x); }
  __device__ static void unpack(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct El<float> {
  static constexpr int kVec = 4;
  __device__ static float get(const float* p, long long i) { return p[i]; }
  __device__ static void put(float* p, long long i, float x) { p[i] = x; }
  __device__ static void unpack(uint4 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// A chunk of one rope part: pairs [i0, i0 + n) as (x_i, x_{i+R/2}); n is the
// vector width on the vector path and 1 on the element path.
template <typename T>
struct Chunk {
  static constexpr int V = El<T>::kVec;
  uint4 a, b;    // vector path: the two halves' 16-byte pieces
  float lo, hi;  // element path
  __device__ void load(const T* src, int R, int vec, int item) {
    const int h = R / 2;
    if (vec) {
      a = *reinterpret_cast<const uint4*>(src + item * V);
      b = *reinterpret_cast<const uint4*>(src + h + item * V);
    } else {
      lo = El<T>::get(src, item);
      hi = El<T>::get(src, h + item);
    }
  }
  // turn pair i by the angle whose cosine and sine are cs[i], sn[i]
  __device__ void store(T* dst, int R, int vec, int item, const float* cs, const float* sn) const {
    const int h = R / 2;
    if (vec) {
      const int i0 = item * V;
      float x0[V], x1[V], y0[V], y1[V];
      El<T>::unpack(a, x0);
      El<T>::unpack(b, x1);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const float c = cs[i0 + j], s = sn[i0 + j];
        y0[j] = fmaf(x0[j], c, -x1[j] * s);
        y1[j] = fmaf(x1[j], c, x0[j] * s);
      }
      *reinterpret_cast<uint4*>(dst + i0) = El<T>::pack(y0);
      *reinterpret_cast<uint4*>(dst + h + i0) = El<T>::pack(y1);
    } else {
      const float c = cs[item], s = sn[item];
      El<T>::put(dst, item, fmaf(lo, c, -hi * s));
      El<T>::put(dst, h + item, fmaf(hi, c, lo * s));
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) k_rope_append(const RopeArgs a) {
  __shared__ float s_cos[kMaxHalf], s_sin[kMaxHalf];
  const int b = blockIdx.x / a.Q, t = blockIdx.x % a.Q;
  const int tid = threadIdx.x;
  const int half = a.R / 2;
  const int per_row = a.vec ? half / El<T>::kVec : half;  // chunks per rope part
  const int CR = a.C + a.R;
  const long long qrow = ((long long)b * a.Q + t) * a.H;
  const T* qi = static_cast<const T*>(a.q_in) + qrow * a.R;
  T* qo = static_cast<T*>(a.q_out) + qrow * a.R;
  const T* src = static_cast<const T*>(a.kv_new) + ((long long)b * a.Q + t) * CR;

  // ---- loads that need no position first: this thread's first query chunks
  // and its first piece of the latent row, in flight while the length, the
  // pages and the angles are worked out
  const long long L = a.prefix_len[b];
  const int depth = a.depths[(long long)b * a.Q + t];
  const int n_q = a.H * per_row;
  Chunk<T> qp[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int it = tid + k * kThreads;
    if (it < n_q) qp[k].load(qi + (long long)(it / per_row) * a.R, a.R, a.vec, it % per_row);
  }
  const int n_lat = a.vec ? a.C / El<T>::kVec : a.C;
  uint4 lat_v = make_uint4(0, 0, 0, 0);
  T lat_e{};
  if (tid < n_lat) {
    if (a.vec)
      lat_v = reinterpret_cast<const uint4*>(src)[tid];
    else
      lat_e = src[tid];
  }

  // ---- the sequence's slots [L, L+Q) must lie in its pages and the cache;
  // every CTA of the sequence takes the same decision
  const int32_t* bt = a.block_table + (long long)b * a.max_pages;
  int code = 0;
  if (L < 0 || L + a.Q > (long long)a.max_pages * a.page_size) code = DDT_ST_CAPACITY;
  if (code == 0) {
    bool bad = false;
    for (int s = tid; s < a.Q; s += kThreads) {
      const long long slot = L + s;
      const long long pg = bt[slot / a.page_size];
      const long long row = pg * a.page_size + slot % a.page_size;
      if (pg < 0 || row >= a.kv_rows) bad = true;
    }
    if (__syncthreads_or(bad)) code = DDT_ST_RANGE;
  }
  if (code) {
    if (t == 0 && tid == 0) atomicOr(a.status + b, code);
    return;
  }

  // ---- this slot's angles: position times frequency in double, reduced
  // modulo 2*pi with 2*pi split in two doubles (Cody and Waite's additive
  // reduction), then float sine and cosine of the remainder
  const double pos = (double)(L + (depth > 0 ? depth : 0));
  for (int i = tid; i < half; i += kThreads) {
    const double ang = pos * a.freqs.f[i];
    const double k = rint(ang * 0.15915494309189535);  // 1 / (2*pi)
    double r = fma(-k, 6.283185307179586, ang);         // 2*pi, leading part
    r = fma(-k, 2.4492935982947064e-16, r);             // 2*pi, trailing part
    float s, c;
    sincosf((float)r, &s, &c);
    s_cos[i] = c;
    s_sin[i] = s;
  }
  __syncthreads();

  // ---- the H query rope parts of this slot
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int it = tid + k * kThreads;
    if (it < n_q)
      qp[k].store(qo + (long long)(it / per_row) * a.R, a.R, a.vec, it % per_row, s_cos, s_sin);
  }
  for (int it = tid + kPre * kThreads; it < n_q; it += kThreads) {
    Chunk<T> c;
    c.load(qi + (long long)(it / per_row) * a.R, a.R, a.vec, it % per_row);
    c.store(qo + (long long)(it / per_row) * a.R, a.R, a.vec, it % per_row, s_cos, s_sin);
  }

  // ---- the latent row to cache slot L + t: latent part copied, rope part turned
  const long long slot = L + t;
  long long row = (long long)bt[slot / a.page_size] * a.page_size + slot % a.page_size;
  if (!DDT_GUARD(row >= 0 && row < a.kv_rows, 601, a.status + b)) return;
  T* dst = static_cast<T*>(a.kv) + row * CR;
  if (a.vec) {
    if (tid < n_lat) reinterpret_cast<uint4*>(dst)[tid] = lat_v;
    for (int it = tid + kThreads; it < n_lat; it += kThreads)
      reinterpret_cast<uint4*>(dst)[it] = reinterpret_cast<const uint4*>(src)[it];
  } else {
    if (tid < n_lat) dst[tid] = lat_e;
    for (int it = tid + kThreads; it < n_lat; it += kThreads) dst[it] = src[it];
  }
  for (int it = tid; it < per_row; it += kThreads) {
    Chunk<T> c;
    c.load(src + a.C, a.R, a.vec, it);
    c.store(dst + a.C, a.R, a.vec, it, s_cos, s_sin);
  }
}

}  // namespace

cudaError_t launch_rope_append(const ddt_attn_dims& d, const RopeFreqs& freqs,
                               const int32_t* depths, const int32_t* prefix_len,
                               const int32_t* block_table, const void* q_in, void* q_out,
                               const void* kv_new, void* kv, int32_t* status,
                               cudaStream_t stream) {
  RopeArgs a;
  a.B = d.B;
  a.Q = d.Q;
  a.H = d.H;
  a.C = d.C;
  a.R = d.R;
  a.page_size = d.page_size;
  a.max_pages = d.max_pages;
  a.kv_rows = d.kv_rows;
  a.depths = depths;
  a.prefix_len = prefix_len;
  a.block_table = block_table;
  a.q_in = q_in;
  a.q_out = q_out;
  a.kv_new = kv_new;
  a.kv = kv;
  a.status = status;
  a.freqs = freqs;
  const int esize = d.dtype == DDT_BF16 ? 2 : 4;
  const int vw = 16 / esize;
  const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  a.vec = (d.R / 2) % vw == 0 && d.C % vw == 0 && al(q_in) && al(q_out) && al(kv_new) && al(kv);
  const long long grid = (long long)d.B * d.Q;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d.dtype == DDT_BF16)
    k_rope_append<__nv_bfloat16><<<(unsigned)grid, kThreads, 0, stream>>>(a);
  else
    k_rope_append<float><<<(unsigned)grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ddt
