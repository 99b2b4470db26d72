// B. Tree-verify MLA-absorb attention on the Blackwell tensor cores (bf16 in,
// fp32 accumulate in TMEM).
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": verify attention in MLA absorb form, tree [verified_id, drafts]
// at cache positions L + depth, mask [ones over the prefix | visibility];
// "The Milestone Commit", section "Input Knowledge Required": the latent
// cache of Kimi K2.6 (kv_lora_rank 512, plus a 64-wide rope part).
//
// Per sequence the Q*H query rows (row = query position * H + head) share one
// latent KV head, so QK^T and PV are dense contractions:
//   S = [q_lat | q_pe] . [c_kv | k_pe]^T   (contraction 576)
//   O = softmax(S * scale, masked) . c_kv  (output 512)
// An fp32 O for 128 rows x 512 columns fills all 512 TMEM columns of an SM,
// leaving nothing for S. So two CTAs of a cluster share one 128-row tile:
// CTA h owns contraction dims [256h, 256h+256) of c_kv plus [32h, 32h+32) of
// the rope part, and output dims [256h, 256h+256). Each computes a partial S
// over its 288 dims on the tensor cores, sends it to its peer through
// distributed shared memory and adds the peer's; both CTAs then hold the
// same S bit for bit (fp32 addition commutes), run the same online softmax,
// and accumulate their own half of O. No FLOP is done twice.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 issues tcgen05
// MMAs and owns the TMEM allocation, warps 2-5 (one thread per query row)
// run the softmax and the epilogue. KV tiles of 64 keys are double
// buffered; S is double buffered in TMEM so the QK^T of tile j+1 runs while
// the softmax of tile j does. The key range of a sequence can be split over
// several clusters (split-KV); partial results are merged by k_combine.
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>

#include <cudaTypedefs.h>

#include "ddt_internal.cuh"
#include "sm100_ptx.cuh"

namespace ddt {
namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 64;   // keys per KV tile
constexpr int kC = 512;
constexpr int kR = 64;
constexpr int kThreads = 192;

constexpr uint32_t kQChunkBytes = kBM * 128;   // 64 dims x 128 rows, 128-byte swizzle
constexpr uint32_t kQRopeBytes = kBM * 64;     // 32 dims x 128 rows, 64-byte swizzle
constexpr uint32_t kKVChunkBytes = kBN * 128;  // 64 dims x 64 keys
constexpr uint32_t kKVRopeBytes = kBN * 64;    // 32 dims x 64 keys
constexpr uint32_t kStageBytes = 4 * kKVChunkBytes + kKVRopeBytes;
constexpr uint32_t kQBytes = 4 * kQChunkBytes + kQRopeBytes;
constexpr uint32_t kRecvStride = kBN * 4 + 16;  // padded: row r at r * 272 bytes

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_QROPE = 4 * kQChunkBytes;
constexpr uint32_t OFF_KV = OFF_QROPE + kQRopeBytes;
constexpr uint32_t OFF_RECV = OFF_KV + 2 * kStageBytes;
constexpr uint32_t OFF_P = OFF_RECV + kBM * kRecvStride;
constexpr uint32_t OFF_BAR = OFF_P + kBM * 128;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0, "swizzled buffers need 1 KB alignment");
static_assert(kStageBytes % 1024 == 0, "stage size");

enum Bar {
  B_Q_FULL = 0,
  B_KV_FULL = 1,   // +stage
  B_KV_EMPTY = 3,  // +stage
  B_S_FULL = 5,    // +buffer
  B_S_EMPTY = 7,   // +buffer
  B_P_FULL = 9,
  B_PV_DONE = 10,
  B_RECV_FULL = 11,
  B_SEND_OK = 12,
  B_MMA_DONE = 13,
  N_BARS = 14
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;  // O half at columns [256, 512); S buffers at [0,64), [64,128)

constexpr uint32_t kIdescS = idesc_bf16_f32(128, kBN, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, true);

struct Params {
  int B, Q, H;
  int page_size, max_pages;
  long long kv_rows;
  float scale_log2;
  int n_rt, n_split;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const unsigned long long* vis_bits;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  float* part_o;
  float* part_lse;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// rows of this CTA's half written as zero (capacity/range errors, empty splits)
__device__ void write_empty(const Params& p, int b, int rt, int sp, uint32_t rank) {
  const int QH = p.Q * p.H;
  const long long total = (long long)p.B * QH;
  for (int e = threadIdx.x; e < kBM * 32; e += kThreads) {
    const int r = e >> 5, c = e & 31;  // 32 chunks of 8 columns per half row
    const int lr = (int)rt * kBM + r;
    if (lr >= QH) continue;
    const long long grow = (long long)b * QH + lr;
    if (p.n_split == 1) {
      reinterpret_cast<uint4*>(p.out + grow * kC + 256 * rank)[c] = make_uint4(0, 0, 0, 0);
      if (rank == 0 && c == 0 && p.lse) p.lse[grow] = -INFINITY;
    } else {
      float4* dst = reinterpret_cast<float4*>(p.part_o + ((long long)sp * total + grow) * kC +
                                              256 * rank);
      dst[2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
      dst[2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rank == 0 && c == 0) p.part_lse[(long long)sp * total + grow] = -INFINITY;
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_verify_attn_bf16(const __grid_constant__ CUtensorMap tm_kv_c,
                       const __grid_constant__ CUtensorMap tm_kv_r,
                       const __grid_constant__ CUtensorMap tm_q_c,
                       const __grid_constant__ CUtensorMap tm_q_r, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  // 1 KB alignment for the swizzled tiles
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + N_BARS * 8);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const long long unit = blockIdx.x >> 1;
  const int sp = (int)(unit % p.n_split);
  const int rt = (int)((unit / p.n_split) % p.n_rt);
  const int b = (int)(unit / ((long long)p.n_split * p.n_rt));
  const int QH = p.Q * p.H;
  const long long total_rows = (long long)p.B * QH;
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;

  // ---- capacity and page checks: identical decision in both CTAs ---------
  const long long L = p.prefix_len[b];
  const long long n_keys = L + p.Q;
  int code = 0;
  if (L < 0 || n_keys > (long long)p.max_pages * p.page_size) code = DDT_ST_CAPACITY;
  if (code == 0) {
    const long long n_pages = (n_keys + p.page_size - 1) / p.page_size;
    const long long kv_pages = p.kv_rows / p.page_size;
    bool badp = false;
    for (long long q = tid; q < n_pages; q += kThreads) {
      const long long pg = bt[q];
      if (pg < 0 || pg >= kv_pages) badp = true;
    }
    if (__syncthreads_or(badp)) code = DDT_ST_RANGE;
  }
  const int n_tiles = (int)((n_keys + kBN - 1) / kBN);
  const int tps = (n_tiles + p.n_split - 1) / p.n_split;
  const int j_begin = sp * tps;
  const int nt = code ? 0 : max(0, min(n_tiles, j_begin + tps) - j_begin);
  if (nt == 0) {
    write_empty(p, b, rt, sp, rank);
    if (code && rt == 0 && sp == 0 && rank == 0 && tid == 0) atomicOr(p.status + b, code);
    return;  // both CTAs of the cluster take this branch together
  }

  // ---- setup ---------------------------------------------------------------
  if (tid == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_S_EMPTY + s), 4);  // one arrival per softmax warp
    }
    mbar_init(bar(B_P_FULL), 4);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_RECV_FULL), 1);  // local expect_tx; the peer's bytes complete it
    mbar_init(bar(B_SEND_OK), 4);    // the peer's softmax warps
    mbar_init(bar(B_MMA_DONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  cluster_sync();  // the peer's barriers are initialised before any remote arrive

  bool failed = false;
  const long long row0 = (long long)b * QH + (long long)rt * kBM;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      prefetch_tmap(&tm_kv_c);
      prefetch_tmap(&tm_kv_r);
      mbar_expect_tx(bar(B_Q_FULL), kQBytes);
      for (int c = 0; c < 4; ++c)
        tma_load_2d(sbase + OFF_Q + c * kQChunkBytes, &tm_q_c, 256 * rank + 64 * c, (int)row0,
                    bar(B_Q_FULL));
      tma_load_2d(sbase + OFF_QROPE, &tm_q_r, 32 * rank, (int)row0, bar(B_Q_FULL));
      int issued = 0;
      for (int jj = 0; jj < nt; ++jj) {
        const int s = jj & 1;
        if (jj >= 2 && !mbar_wait(bar(B_KV_EMPTY + s), ((jj >> 1) - 1) & 1)) {
          failed = true;
          break;
        }
        const long long t0 = (long long)(j_begin + jj) * kBN;
        const long long krow = (long long)bt[t0 / p.page_size] * p.page_size + t0 % p.page_size;
        const uint32_t st = sbase + OFF_KV + s * kStageBytes;
        mbar_expect_tx(bar(B_KV_FULL + s), kStageBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(st + c * kKVChunkBytes, &tm_kv_c, 256 * rank + 64 * c, (int)krow,
                      bar(B_KV_FULL + s));
        tma_load_2d(st + 4 * kKVChunkBytes, &tm_kv_r, kC + 32 * rank, (int)krow,
                    bar(B_KV_FULL + s));
        ++issued;
      }
      // no copy may still be landing in shared memory when the CTA leaves
      for (int jj = max(0, issued - 2); jj < issued; ++jj)
        if (!mbar_wait(bar(B_KV_FULL + (jj & 1)), (jj >> 1) & 1)) failed = true;
      if (!mbar_wait(bar(B_Q_FULL), 0)) failed = true;
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t p_desc_base = sbase + OFF_P;
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(bar(B_P_FULL), t & 1)) return false;
        tc_fence_after();
        const uint32_t st = sbase + OFF_KV + (t & 1) * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t ad = smem_desc(p_desc_base + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(st + kk * 2048, kKVChunkBytes, 1024, kSwizzle128B);
          umma_bf16(tmem + kTmemO, ad, bd, kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_PV_DONE));
        umma_commit(bar(B_KV_EMPTY + (t & 1)));
        return true;
      };
      if (!mbar_wait(bar(B_Q_FULL), 0)) failed = true;
      for (int jj = 0; jj < nt && !failed; ++jj) {
        const int s = jj & 1;
        if (!mbar_wait(bar(B_KV_FULL + s), (jj >> 1) & 1)) { failed = true; break; }
        if (jj >= 2 && !mbar_wait(bar(B_S_EMPTY + s), ((jj >> 1) - 1) & 1)) { failed = true; break; }
        tc_fence_after();
        const uint32_t st = sbase + OFF_KV + s * kStageBytes;
        const uint32_t d = tmem + s * kBN;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad =
                smem_desc(sbase + OFF_Q + c * kQChunkBytes + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd =
                smem_desc(st + c * kKVChunkBytes + kk * 32, 16, 1024, kSwizzle128B);
            umma_bf16(d, ad, bd, kIdescS, (c | kk) ? 1u : 0u);
          }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t ad = smem_desc(sbase + OFF_QROPE + kk * 32, 16, 512, kSwizzle64B);
          const uint64_t bd = smem_desc(st + 4 * kKVChunkBytes + kk * 32, 16, 512, kSwizzle64B);
          umma_bf16(d, ad, bd, kIdescS, 1u);
        }
        umma_commit(bar(B_S_FULL + s));
        if (jj >= 1 && !issue_pv(jj - 1)) { failed = true; break; }
      }
      if (!failed && !issue_pv(nt - 1)) failed = true;
      // every MMA issued above has completed before TMEM is released
      umma_commit(bar(B_MMA_DONE));
      if (!mbar_wait(bar(B_MMA_DONE), 0)) failed = true;
    }
  } else {
    // ======================= softmax + epilogue =======================
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
    const int lr = rt * kBM + r;
    const bool row_ok = lr < QH;
    const int qi = row_ok ? lr / p.H : 0;
    const int W = (p.Q + 63) >> 6;
    unsigned long long vis0 = 0ull, vis1 = 0ull;
    if (row_ok) {
      const unsigned long long* vb = p.vis_bits + ((size_t)b * p.Q + qi) * W;
      vis0 = vb[0];
      if (W > 1) vis1 = vb[1];
    }
    const uint32_t recv_local = sbase + OFF_RECV + r * kRecvStride;
    const uint32_t recv_remote = map_peer(recv_local, peer);
    const uint32_t recv_full_remote = map_peer(bar(B_RECV_FULL), peer);  // st.async target
    const uint32_t send_ok_remote = map_peer(bar(B_SEND_OK), peer);
    const uint32_t p_row = sbase + OFF_P + (r >> 3) * 1024 + (r & 7) * 128;

    constexpr uint32_t kRecvBytes = kBM * kBN * 4;  // one partial S tile
    if (tid == 64) mbar_expect_tx(bar(B_RECV_FULL), kRecvBytes);
    float m_run = -INFINITY, l_run = 0.f;
    for (int jj = 0; jj < nt; ++jj) {
      const int s = jj & 1;
      const long long t0 = (long long)(j_begin + jj) * kBN;
      // waits are made warp-uniform: the tcgen05 loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S_FULL + s), (jj >> 1) & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld32(t_lane + s * kBN, lo);
        tmem_ld32(t_lane + s * kBN + 32, hi);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_EMPTY + s));

      // exchange partial scores with the peer CTA (one row per thread)
      if (jj >= 1 &&
          !__all_sync(0xffffffffu, mbar_wait_cluster(bar(B_SEND_OK), (jj - 1) & 1))) {
        failed = true;
        break;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        st_async_v4(recv_remote + 16 * k, sv[4 * k], sv[4 * k + 1], sv[4 * k + 2],
                    sv[4 * k + 3], recv_full_remote);
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar(B_RECV_FULL), jj & 1))) {
        failed = true;
        break;
      }
      // arm the next phase before telling the peer it may send again
      if (tid == 64 && jj + 1 < nt) mbar_expect_tx(bar(B_RECV_FULL), kRecvBytes);
      float x[64];
      const float4* rv = reinterpret_cast<const float4*>(smem + OFF_RECV + r * kRecvStride);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float4 o4 = rv[k];
        x[4 * k + 0] = (__uint_as_float(sv[4 * k + 0]) + o4.x) * p.scale_log2;
        x[4 * k + 1] = (__uint_as_float(sv[4 * k + 1]) + o4.y) * p.scale_log2;
        x[4 * k + 2] = (__uint_as_float(sv[4 * k + 2]) + o4.z) * p.scale_log2;
        x[4 * k + 3] = (__uint_as_float(sv[4 * k + 3]) + o4.w) * p.scale_log2;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(send_ok_remote);

      // mask: keys past the prefix are visible only along the ancestor path
      if (t0 + kBN > L) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const long long slot = t0 + k;
          bool vis = slot < L;
          if (!vis && slot < n_keys) {
            const int t = (int)(slot - L);
            vis = ((t < 64 ? vis0 : vis1) >> (t & 63)) & 1ull;
          }
          if (!vis) x[k] = -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx8[q] = x[q];
#pragma unroll
      for (int k = 8; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], x[k]);
      const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // lazy rescale: the reference max moves only when the row max passes it by 8 (x2^8)
      float factor = 1.f;
      bool rescale = false;
      if (mt > m_run + 8.f) {
        factor = ex2(m_run - mt);  // 0 when m_run is -inf
        l_run *= factor;
        rescale = jj > 0;
        m_run = mt;
      }
      uint32_t pk[32];
      float ls8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const float m_use = m_run == -INFINITY ? 0.f : m_run;  // every x is -inf then: p = 0
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2(x[2 * k] - m_use);
        const float p1 = ex2(x[2 * k + 1] - m_use);
        pk[k] = pack_bf16(p0, p1);
        const __nv_bfloat162 pb = *reinterpret_cast<__nv_bfloat162*>(&pk[k]);
        ls8[k & 7] += __low2float(pb) + __high2float(pb);
      }
      l_run += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));

      // keys past the end of the sequence in the last tile: zero their values
      // so that 0 * (whatever the page holds) cannot turn into NaN
      if (t0 + kBN > n_keys && r < kBN && t0 + r >= n_keys) {
        const uint32_t st = OFF_KV + s * kStageBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4* rowp = reinterpret_cast<uint4*>(smem + st + c * kKVChunkBytes +
                                                 (r >> 3) * 1024 + (r & 7) * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q) rowp[q] = make_uint4(0, 0, 0, 0);
        }
      }
      // P buffer and O are free once PV of the previous tile has completed
      if (jj >= 1) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_PV_DONE), (jj - 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
      }
      // rows that keep their reference max multiply by 1; the TMEM round trip
      // is done by the whole warp whenever any of its rows needs it
      if (__any_sync(0xffffffffu, rescale)) {
        if (!rescale) factor = 1.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t ov[32];
          tmem_ld32(t_lane + kTmemO + 32 * c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * factor);
          tmem_st32(t_lane + kTmemO + 32 * c, ov);
        }
        tmem_st_wait();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = p_row + ((uint32_t)(c ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL));
    }

    // ---- epilogue: O half / l ------------------------------------------------
    if (!__all_sync(0xffffffffu, !failed && mbar_wait(bar(B_PV_DONE), (nt - 1) & 1)))
      failed = true;
    if (!failed) {
      tc_fence_after();
      const bool live = l_run > 0.f;
      const float inv_l = live ? 1.f / l_run : 0.f;
      const float lse_v = live ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
      const long long grow = row0 + r;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_lane + kTmemO + 32 * c, ov);
        tmem_ld_wait();
        if (!row_ok) continue;
        if (p.n_split == 1) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + grow * kC + 256 * rank + 32 * c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            dst[q] = make_uint4(pack_bf16(__uint_as_float(ov[8 * q + 0]) * inv_l,
                                          __uint_as_float(ov[8 * q + 1]) * inv_l),
                                pack_bf16(__uint_as_float(ov[8 * q + 2]) * inv_l,
                                          __uint_as_float(ov[8 * q + 3]) * inv_l),
                                pack_bf16(__uint_as_float(ov[8 * q + 4]) * inv_l,
                                          __uint_as_float(ov[8 * q + 5]) * inv_l),
                                pack_bf16(__uint_as_float(ov[8 * q + 6]) * inv_l,
                                          __uint_as_float(ov[8 * q + 7]) * inv_l));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.part_o + ((long long)sp * total_rows + grow) * kC + 256 * rank + 32 * c);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(ov[4 * q + 0]) * inv_l,
                                 __uint_as_float(ov[4 * q + 1]) * inv_l,
                                 __uint_as_float(ov[4 * q + 2]) * inv_l,
                                 __uint_as_float(ov[4 * q + 3]) * inv_l);
        }
      }
      if (row_ok && rank == 0) {
        if (p.n_split == 1) {
          if (p.lse) p.lse[grow] = lse_v;
        } else {
          p.part_lse[(long long)sp * total_rows + grow] = lse_v;
        }
      }
    }
  }

  if (failed) atomicOr(p.status + b, DDT_ST_TIMEOUT);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // no remote store or arrive may target a CTA that has left
}

// Merge of the split-KV partials: o = sum_s w_s o_s / sum_s w_s with
// w_s = exp(lse_s - max lse); one warp per query row, 16 columns per lane.
__global__ void __launch_bounds__(256) k_combine(long long total_rows, int n_split,
                                                 const float* __restrict__ part_o,
                                                 const float* __restrict__ part_lse,
                                                 __nv_bfloat16* __restrict__ out,
                                                 float* __restrict__ lse_out) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= total_rows) return;
  float m = -INFINITY;
  for (int s = 0; s < n_split; ++s) m = fmaxf(m, part_lse[(long long)s * total_rows + row]);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float ls = part_lse[(long long)s * total_rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      wsum += w;
      const float4* src =
          reinterpret_cast<const float4*>(part_o + ((long long)s * total_rows + row) * kC) +
          lane * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = src[q];
        acc[4 * q + 0] = fmaf(w, v.x, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(out + row * kC) + lane * 2;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    dst[q] = make_uint4(pack_bf16(acc[8 * q + 0] * inv, acc[8 * q + 1] * inv),
                        pack_bf16(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                        pack_bf16(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                        pack_bf16(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
  if (lse_out && lane == 0) lse_out[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

// ---------------------------------------------------------------- host side

struct Plan {
  int n_rt, n_split;
  long long units;
};

int sm_count() {
  static int cached[64] = {};
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return n;
  if (cached[dev] == 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    cached[dev] = n;
  return cached[dev] ? cached[dev] : n;
}

// Split of the key range so that clusters fill whole waves: a cluster takes
// two SMs, a wave is sm_count/2 clusters; cost ~ waves * (tiles per unit +
// fixed overhead), plus a merge pass when the range is split.
Plan make_plan(const ddt_attn_dims& d) {
  Plan pl;
  const long long QH = (long long)d.Q * d.H;
  pl.n_rt = (int)((QH + kBM - 1) / kBM);
  const long long base = (long long)d.B * pl.n_rt;
  const long long max_len = d.max_len > d.Q ? d.max_len : d.Q;
  const long long n_tiles = (max_len + kBN - 1) / kBN;
  const long long per_wave = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
  double best = 1e300;
  pl.n_split = 1;
  for (long long s = 1; s <= 64 && s <= n_tiles; ++s) {
    const long long units = base * s;
    const long long waves = (units + per_wave - 1) / per_wave;
    const double cost = (double)waves * (double)((n_tiles + s - 1) / s + 4) + (s > 1 ? 3.0 + s : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      pl.n_split = (int)s;
    }
  }
  pl.units = base * pl.n_split;
  return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swz) {
  auto fn = encoder();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t verify_attn_bf16_workspace(const ddt_attn_dims& d) {
  const Plan pl = make_plan(d);
  if (pl.n_split <= 1) return 0;
  const size_t rows = (size_t)d.B * d.Q * d.H;
  const size_t bytes = (size_t)pl.n_split * rows * (kC * sizeof(float) + sizeof(float));
  return (bytes + 255) & ~size_t(255);
}

cudaError_t launch_verify_attn_bf16(const ddt_attn_dims& d, const void* q_lat, const void* q_pe,
                                    const void* kv, const int32_t* block_table,
                                    const int32_t* prefix_len, const uint64_t* vis_bits,
                                    void* out, float* lse, int32_t* status, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  const Plan pl = make_plan(d);
  const long long rows = (long long)d.B * d.Q * d.H;
  if (d.kv_rows < 1 || rows > 0x7fffffffLL || d.kv_rows > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  CUtensorMap tm_kv_c, tm_kv_r, tm_q_c, tm_q_r;
  const uint64_t row_kv = (kC + kR) * 2;
  if (!encode_2d(&tm_kv_c, kv, kC + kR, (uint64_t)d.kv_rows, row_kv, 64, kBN,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_kv_r, kv, kC + kR, (uint64_t)d.kv_rows, row_kv, 32, kBN,
                 CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_2d(&tm_q_c, q_lat, kC, (uint64_t)rows, kC * 2, 64, kBM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_q_r, q_pe, kR, (uint64_t)rows, kR * 2, 32, kBM, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;

  Params p;
  p.B = d.B; p.Q = d.Q; p.H = d.H;
  p.page_size = d.page_size; p.max_pages = d.max_pages; p.kv_rows = d.kv_rows;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.n_rt = pl.n_rt; p.n_split = pl.n_split;
  p.block_table = block_table; p.prefix_len = prefix_len;
  p.vis_bits = reinterpret_cast<const unsigned long long*>(vis_bits);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse; p.status = status;
  p.part_o = nullptr; p.part_lse = nullptr;
  if (pl.n_split > 1) {
    p.part_o = static_cast<float*>(workspace);
    p.part_lse = p.part_o + (size_t)pl.n_split * rows * kC;
  }
  static int smem_set[64] = {};
  cudaError_t e = ensure_smem_limit(k_verify_attn_bf16, (int)kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  k_verify_attn_bf16<<<(unsigned)(pl.units * 2), kThreads, kSmemBytes, stream>>>(
      tm_kv_c, tm_kv_r, tm_q_c, tm_q_r, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || pl.n_split == 1) return e;
  k_combine<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(rows, pl.n_split, p.part_o,
                                                            p.part_lse, p.out, lse);
  return cudaGetLastError();
}

}  // namespace ddt
