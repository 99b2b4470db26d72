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
// and shared memory cannot also hold Q, so one SM cannot own a 128-row tile.
// Two CTAs of a cluster share it with different roles:
//   * the S-CTA (cluster rank 0) keeps all of Q in TMEM (288 columns, bf16
//     pairs), computes S = QK^T for 64 keys at a time (two TMEM S buffers),
//     runs the online softmax and ships P (bf16, 16 KB per tile) plus the
//     per-row rescale factors to its peer with one bulk shared-memory copy;
//   * the O-CTA (rank 1) keeps O (128 x 512 fp32) in TMEM, loads the c_kv
//     half of each KV tile and accumulates O += P V; its row warps apply the
//     (rare) rescales and write the output.
// No FLOP is done twice. The peer-to-peer traffic is P only (bf16, one way),
// which the cluster link moves in less time than the S-CTA spends on QK^T.
//
// Warp roles (224 threads): warp 0 issues TMA loads; warp 1 owns the TMEM
// allocation and issues tcgen05 MMAs; warps 2-5 handle one query row per
// thread; in the S-CTA warp 6 is a second MMA issuer (a single thread issues
// an MMA only about every 50 cycles, slower than an N=64 MMA runs, so the two
// issuers take alternate key tiles). Q reaches the S-CTA by TMA (staged in
// the ring, then copied to TMEM by the row warps). Each CTA fetches a 64-key
// tile with ONE TMA request (the TMA engine costs about 500 cycles per
// request whatever its size, so small boxes starve the tensor cores): a 3-D
// tensor map views the cache as {64 dims, keys, 9 chunks} with strides (row,
// 128 B), and a box of {64, 64, 9} (S-CTA, 72 KB) or {64, 64, 8} (O-CTA, c_kv
// only, 64 KB) lands as per-chunk 64-key x 128-byte swizzled tiles. Two
// stages per CTA. The O-CTA writes its output rows through shared memory with
// one bulk copy per row. The key range of a sequence can be split over
// several clusters (split-KV); partial results are merged by k_combine.
#include <cuda_bf16.h>
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "ddt_internal.cuh"
#include "sm100_ptx.cuh"
#include "tree_build_warp.cuh"

namespace ddt {
DDT_CHECKS_FILE(bf16)
namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 64;   // keys per KV tile
constexpr int kC = 512;
constexpr int kR = 64;
constexpr int kThreads = 224;

constexpr uint32_t kChunkBytes = kBN * 128;             // 64 keys x 64 dims, 128-byte swizzle
constexpr int kChunksPerTile = (kC + kR) / 64;          // 9 (8 c_kv + 1 rope)
constexpr uint32_t kTileS = kChunksPerTile * kChunkBytes;  // S-CTA stage: 72 KB
constexpr uint32_t kTileO = 8 * kChunkBytes;               // O-CTA stage: c_kv, 64 KB
constexpr uint32_t kHalfBytes = 4 * kChunkBytes;           // 256 c_kv dims x 64 keys
constexpr int kStages = 2;
constexpr int kMsgSlots = 4;  // P messages in flight between the two CTAs
constexpr uint32_t kPBytes = kBM * 128;                 // P tile: 128 rows x 64 keys bf16
constexpr uint32_t kMsgBytes = kPBytes + kBM * 4 + 16;  // P | per-row factor | 4 warp flags
constexpr uint32_t kMsgStride = 17408;                  // 1 KB aligned message slots
constexpr uint32_t kFinBytes = kBM * 4;                 // per-row 1/l
constexpr uint32_t kQBytes = kBM * (kC + kR) * 2;       // Q tile: 128 rows x 576 bf16
constexpr uint32_t kOutStride = 1040;                   // staged output row: 1 KB + 16 B

// S-CTA shared memory
constexpr uint32_t S_RING = 0;
constexpr uint32_t S_STAGE = S_RING + kStages * kTileS;  // outgoing messages
constexpr uint32_t S_FIN = S_STAGE + kMsgSlots * kMsgStride;
constexpr uint32_t S_VIS = S_FIN + 1024;  // ancestor words of the fused build [kMaxQ][kMaxW]
constexpr uint32_t S_END = S_VIS + kMaxQ * kMaxW * 8;
// O-CTA shared memory
constexpr uint32_t O_RING = 0;
constexpr uint32_t O_MSG = O_RING + kStages * kTileO;  // incoming messages
constexpr uint32_t O_FIN = O_MSG + kMsgSlots * kMsgStride;
constexpr uint32_t O_BUILD = O_FIN + 1024;  // fused tree build: tb::Smem + staged candidates
constexpr uint32_t kBuildBytes = (uint32_t)tb::smem_bytes(kFuseMaxCand, 1);
constexpr uint32_t O_END = O_BUILD + ((kBuildBytes + 1023) & ~1023u);

// both CTAs: the sequence's block-table row, read once by the page check
constexpr int kBtMax = 1024;  // pages staged (longer rows are read from global memory)
constexpr uint32_t OFF_BT = (S_END > O_END ? S_END : O_END);
constexpr uint32_t OFF_BAR = OFF_BT + kBtMax * 4;
constexpr uint32_t kSmemBytes = OFF_BAR + 1024 + 1024;  // barriers + alignment slack
static_assert(S_STAGE % 1024 == 0 && O_MSG % 1024 == 0 && kMsgStride % 1024 == 0, "alignment");
static_assert(kMsgBytes <= kMsgStride && kMsgBytes % 16 == 0, "message size");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kQBytes <= kStages * kTileS, "the Q tile is staged in the S-CTA ring");
static_assert(kBM * kOutStride <= O_FIN, "the output is staged in the O-CTA ring and messages");
static_assert(offsetof(tb::Smem, anc) % 16 == 0, "ancestor words are bulk-copied");

// mbarriers (indices into one array; each CTA uses its own subset)
enum Bar {
  // S-CTA
  B_RING_FULL = 0,                       // +stage
  B_RING_EMPTY = B_RING_FULL + kStages,  // +stage
  B_S_FULL = B_RING_EMPTY + kStages,     // +buffer
  B_S_EMPTY = B_S_FULL + 2,          // +buffer
  B_Q_TMEM = B_S_EMPTY + 2,
  B_Q_FULL = B_Q_TMEM + 1,  // Q tile landed in the ring (TMA)
  B_P_FREE = B_Q_FULL + 1,  // +message slot; arrived by the O-CTA
  // O-CTA
  B_HALF_FULL = B_P_FREE + kMsgSlots,    // +stage
  B_HALF_EMPTY = B_HALF_FULL + kStages,  // +stage
  B_P_FULL = B_HALF_EMPTY + kStages,     // +message slot; completed by the S-CTA's copy
  B_O_READY = B_P_FULL + kMsgSlots,
  // +message slot: PV of the tile in that slot has completed (one barrier per
  // slot: a barrier cannot complete another phase before the row warps have
  // waited on this one, since its next tile needs the slot back)
  B_PV_DONE = B_O_READY + 1,
  B_FIN_FULL = B_PV_DONE + kMsgSlots,
  B_TAIL_OK = B_FIN_FULL + 1,
  // both
  B_MMA_DONE = B_TAIL_OK + 1,
  B_TREE = B_MMA_DONE + 1,  // S-CTA: ancestor words of the fused build landed
  N_BARS = B_TREE + 1
};
static_assert(N_BARS * 8 + 16 <= 1024, "barrier area");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;    // S-CTA: Q c_kv part [0,256), rope [256,288)
constexpr uint32_t kTmemS = 384;  // S-CTA: S buffers [384,448), [448,512)

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
  const __nv_bfloat16* q_lat;
  const __nv_bfloat16* q_pe;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  __nv_bfloat16* part_o;  // split-KV partial outputs (normalised by their own l)
  float* part_lse;
  int fuse;     // build the tree here (vis_bits unused)
  TreeFuse tf;  // its inputs and outputs
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta,
                                                  uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void row_barrier() {  // the 128 row threads (warps 2-5)
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// Same barrier, returning the AND of `ok` over the 128 row threads, so that a
// bounded wait that gave up in one warp makes all four leave together.
__device__ __forceinline__ bool row_barrier_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

// rows of this unit written as empty (capacity/range errors, empty splits):
// the O-CTA writes zero output, the S-CTA writes lse = -inf
__device__ void write_empty(const Params& p, int b, int rt, int sp, uint32_t rank) {
  const int QH = p.Q * p.H;
  const long long total = (long long)p.B * QH;
  for (int e = threadIdx.x; e < kBM * 64; e += kThreads) {
    const int r = e >> 6, c = e & 63;  // 64 chunks of 8 columns per row
    const int lr = rt * kBM + r;
    if (lr >= QH) continue;
    const long long grow = (long long)b * QH + lr;
    if (rank == 1) {
      if (p.n_split == 1) {
        reinterpret_cast<uint4*>(p.out + grow * kC)[c] = make_uint4(0, 0, 0, 0);
      } else {
        reinterpret_cast<uint4*>(p.part_o + ((long long)sp * total + grow) * kC)[c] =
            make_uint4(0, 0, 0, 0);
      }
    } else if (c == 0) {
      if (p.n_split == 1) {
        if (p.lse) p.lse[grow] = -INFINITY;
      } else {
        p.part_lse[(long long)sp * total + grow] = -INFINITY;
      }
    }
  }
}

// The draft tree of sequence b, built by the calling warp into `bsm`
// (tb::Smem + staged candidates). Returns the node count; *bad as tb::build_warp.
__device__ int fused_build(const TreeFuse& f, int b, unsigned char* bsm, bool* bad) {
  const int De = min(f.D, f.budget), Ke = min(f.K, f.budget);
  tb::Smem& S = *reinterpret_cast<tb::Smem*>(bsm);
  double* s_logp = reinterpret_cast<double*>(bsm + sizeof(tb::Smem));
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_logp + De * Ke);
  const float* lp = f.topk_logp + (size_t)b * f.D * f.K;
  const int32_t* ip = f.topk_ids + (size_t)b * f.D * f.K;
  const int32_t root = f.root_tok[b];
  switch (tb::slots_for(f.budget + 1)) {
    case 1: return tb::build_warp<1>(lp, ip, root, f.D, f.K, f.budget, f.V, De, Ke, S, s_logp, s_ids, bad);
    case 2: return tb::build_warp<2>(lp, ip, root, f.D, f.K, f.budget, f.V, De, Ke, S, s_logp, s_ids, bad);
    case 3: return tb::build_warp<3>(lp, ip, root, f.D, f.K, f.budget, f.V, De, Ke, S, s_logp, s_ids, bad);
    default: return tb::build_warp<4>(lp, ip, root, f.D, f.K, f.budget, f.V, De, Ke, S, s_logp, s_ids, bad);
  }
}
// Tree outputs of sequence b from the build in `bsm`; OR-s the build's status bits.
__device__ void fused_write(const Params& p, int b, const unsigned char* bsm, int n, bool bad) {
  const TreeFuse& f = p.tf;
  const int32_t st = tb::write_warp(*reinterpret_cast<const tb::Smem*>(bsm), b, f.budget + 1, n,
                                    bad, f.tokens, f.parents, f.depths,
                                    reinterpret_cast<unsigned long long*>(f.vis_bits), f.vis,
                                    f.first_child, f.next_sibling, f.n_nodes);
  if ((threadIdx.x & 31) == 0 && st != 0) atomicOr(p.status + b, st);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_verify_attn_bf16(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_ql,
                       const __grid_constant__ CUtensorMap tm_qp, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + N_BARS * 8);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t rank = cluster_rank();  // 0: S-CTA, 1: O-CTA
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
  const long long row0 = (long long)b * QH + (long long)rt * kBM;

  // Q depends on no check: the S-CTA starts its load before anything else
  // (the checks below are dependent global reads), into the ring, which K
  // takes over once Q is in TMEM. A unit that exits early waits for it.
  if (rank == 0 && tid == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    fence_mbar_init();
    mbar_expect_tx(bar(B_Q_FULL), kQBytes);
    tma_load_3d(sbase + S_RING, &tm_ql, 0, (int)row0, 0, bar(B_Q_FULL));
    tma_load_2d(sbase + S_RING + 8 * kBM * 128, &tm_qp, 0, (int)row0, bar(B_Q_FULL));
  }

  // ---- capacity and page checks: identical decision in both CTAs ---------
  const long long L = p.prefix_len[b];
  const long long n_keys = L + p.Q;
  int code = 0;
  if (L < 0 || n_keys > (long long)p.max_pages * p.page_size) code = DDT_ST_CAPACITY;
  if (code == 0) {
    const long long n_pages = (n_keys + p.page_size - 1) / p.page_size;
    const long long kv_pages = p.kv_rows / p.page_size;
    bool badp = false;
    int32_t* s_bt = reinterpret_cast<int32_t*>(smem + OFF_BT);
    for (long long q = tid; q < n_pages; q += kThreads) {
      const int32_t pg = bt[q];
      if (q < kBtMax) s_bt[q] = pg;
      if (pg < 0 || pg >= kv_pages) badp = true;
    }
    if (__syncthreads_or(badp)) code = DDT_ST_RANGE;
  }
  const int n_tiles = (int)((n_keys + kBN - 1) / kBN);
  // the last unit of a split sequence also walks the tree tiles (and builds
  // the tree): the earlier units take the extra tile when the range divides
  const int tps = p.n_split > 1 ? (n_tiles + p.n_split) / p.n_split : n_tiles;
  const int j_begin = sp * tps;
  const int nt = code ? 0 : max(0, min(n_tiles, j_begin + tps) - j_begin);
  // with a fused build, the unit holding the sequence tail of row tile 0
  // writes the tree (unit 0 when the sequence cannot be attended)
  const int sp_last = code ? 0 : (n_tiles - 1) / tps;
  const bool designated = p.fuse && rt == 0 && sp == sp_last;
  if (nt == 0) {
    // nothing may land after exit: a Q load still pending when the bounded
    // wait gives up is reported, as on the main path
    if (rank == 0 && tid == 0 && !mbar_wait(bar(B_Q_FULL), 0)) atomicOr(p.status + b, DDT_ST_TIMEOUT);
    write_empty(p, b, rt, sp, rank);
    if (code && rt == 0 && sp == 0 && rank == 0 && tid == 0) atomicOr(p.status + b, code);
    if (designated && rank == 1 && warp == 6) {
      bool bad = false;
      const int n = fused_build(p.tf, b, smem + O_BUILD, &bad);
      fused_write(p, b, smem + O_BUILD, n, bad);
    }
    return;  // both CTAs of the cluster take this branch together
  }
  // Row tiles of a sequence walk its key tiles from staggered starting points
  // (all clusters reading the same tile at once contend for the same L2
  // lines). Only tiles that lie wholly in the prefix rotate; the tiles that
  // hold tree keys come last, in order, so that the running max is taken
  // over full prefix tiles before the sparse, masked tree tiles (a walk that
  // starts on a tile with a handful of visible keys rescales O again and
  // again), so that a tree built in this kernel is needed as late as
  // possible, and so that the unit's last tile, which holds the sequence
  // tail, stays last. The online softmax does not depend on the order.
  const int n_pure = (int)(L / kBN);  // tiles with no tree key
  const int nrot = max(0, min(j_begin + nt, n_pure) - j_begin);
  // units with tree tiles build the tree themselves (the designated one has)
  const bool builds = p.fuse && nt > nrot;
  const uint32_t vis_bytes = (uint32_t)(p.Q * kMaxW * 8);

  // ---- setup ---------------------------------------------------------------
  if (tid == 0) {
    if (rank == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(bar(B_RING_FULL + s), 1);
        mbar_init(bar(B_RING_EMPTY + s), 1);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(bar(B_S_FULL + s), 1);
        mbar_init(bar(B_S_EMPTY + s), 4);
      }
      for (int s = 0; s < kMsgSlots; ++s) mbar_init(bar(B_P_FREE + s), 1);
      mbar_init(bar(B_Q_TMEM), 4);
      mbar_init(bar(B_MMA_DONE), 2);  // one commit per MMA issuer
      if (builds) {
        mbar_init(bar(B_TREE), 1);
        mbar_expect_tx(bar(B_TREE), vis_bytes);
      }
    } else {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(bar(B_HALF_FULL + s), 1);
        mbar_init(bar(B_HALF_EMPTY + s), 1);
      }
      for (int s = 0; s < kMsgSlots; ++s) {
        mbar_init(bar(B_P_FULL + s), 1);
        mbar_init(bar(B_PV_DONE + s), 1);
      }
      mbar_init(bar(B_O_READY), 4);
      mbar_init(bar(B_FIN_FULL), 1);
      mbar_init(bar(B_TAIL_OK), 1);
      // arm the first incoming messages and the final 1/l vector
      for (int s = 0; s < kMsgSlots && s < nt; ++s) mbar_expect_tx(bar(B_P_FULL + s), kMsgBytes);
      mbar_expect_tx(bar(B_FIN_FULL), kFinBytes);
      mbar_init(bar(B_MMA_DONE), 1);
    }
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
  cluster_sync();  // the peer's barriers are initialised before any remote operation

  bool failed = false;
  // row tiles of a sequence start their walks at most three tiles apart (see
  // the 256-row kernel: spreading the starts over the prefix multiplies the
  // DRAM bytes once the sequences in flight outgrow L2)
  const int rot = nrot > 0 ? (rt % 4) % nrot : 0;
  auto tile_of = [&](int jj) -> int {
    return (jj < nrot) ? j_begin + (jj + rot) % nrot : j_begin + jj;
  };
  auto krow_of = [&](int jj) -> long long {
    const long long t0 = (long long)tile_of(jj) * kBN;
    const long long pi = t0 / p.page_size;
    if (!DDT_GUARD(pi >= 0 && pi < p.max_pages, 201, p.status + b)) return 0;
    const int32_t pg = pi < kBtMax ? reinterpret_cast<const int32_t*>(smem + OFF_BT)[pi] : bt[pi];
    const long long row = (long long)pg * p.page_size + t0 % p.page_size;
    // a key tile must lie inside the cache (the TMA is clamped to row 0 otherwise)
    return DDT_GUARD(row >= 0 && row + kBN <= p.kv_rows, 202, p.status + b) ? row : 0;
  };

  if (rank == 0) {
    // ========================= S-CTA =========================
    if (warp == 0) {
      if (lane == 0) {
        prefetch_tmap(&tm_s);
        int u = 0;
        // K may overwrite the ring once Q is in TMEM; the Q copy has always
        // landed before anything else is issued (or the CTA leaves)
        if (!mbar_wait(bar(B_Q_TMEM), 0)) failed = true;
        if (!mbar_wait(bar(B_Q_FULL), 0)) failed = true;
        for (; u < nt && !failed; ++u) {  // one 72 KB request per tile
          const int slot = u % kStages;
          if (u >= kStages && !mbar_wait(bar(B_RING_EMPTY + slot), ((u / kStages) - 1) & 1)) {
            failed = true;
            break;
          }
          mbar_expect_tx(bar(B_RING_FULL + slot), kTileS);
          tma_load_3d(sbase + S_RING + slot * kTileS, &tm_s, 0, (int)krow_of(u), 0,
                      bar(B_RING_FULL + slot));
        }
        for (int v = max(0, u - kStages); v < u; ++v)  // nothing may land after the CTA leaves
          if (!mbar_wait(bar(B_RING_FULL + v % kStages), (v / kStages) & 1)) failed = true;
      }
    } else if (warp == 1 || warp == 6) {
      // QK^T: A = Q from TMEM, B = KV chunk (K-major). One thread issues a
      // tcgen05.mma about every 50 cycles, while an N=64 MMA runs in 32, so
      // two issuers take alternate tiles (and own S buffer / ring slot
      // tile & 1) to keep the tensor pipe full.
      if (lane == 0) {
        const int first = warp == 1 ? 0 : 1;
        if (!mbar_wait(bar(B_Q_TMEM), 0)) failed = true;
        tc_fence_after();
        for (int jj = first; jj < nt && !failed; jj += 2) {
          const int sb = jj & 1;
          if (jj >= 2 && !mbar_wait(bar(B_S_EMPTY + sb), ((jj >> 1) - 1) & 1)) {
            failed = true;
            break;
          }
          const uint32_t d = tmem + kTmemS + sb * kBN;
          const int slot = jj % kStages;
          if (!mbar_wait(bar(B_RING_FULL + slot), (jj / kStages) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + S_RING + slot * kTileS;
#pragma unroll
          for (int c = 0; c < kChunksPerTile; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = smem_desc(st + c * kChunkBytes + kk * 32, 16, 1024, kSwizzle128B);
              umma_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * kk, bd, kIdescS, (c | kk) ? 1u : 0u);
            }
          }
          umma_commit(bar(B_RING_EMPTY + slot));
          umma_commit(bar(B_S_FULL + sb));
        }
        umma_commit(bar(B_MMA_DONE));
        if (!mbar_wait(bar(B_MMA_DONE), 0)) failed = true;
      }
    } else {
      // ---------------- softmax (one query row per thread) ----------------
      const int qd = warp & 3;
      const int r = qd * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
      const int lr = rt * kBM + r;
      const bool row_ok = lr < QH;
      const int qi = row_ok ? lr / p.H : 0;
      const int W = (p.Q + 63) >> 6;
      unsigned long long vis0 = 0ull, vis1 = 0ull;
      bool vis_ready = !p.fuse;  // a fused build delivers them before the first tree tile
      if (!p.fuse && row_ok) {
        const unsigned long long* vb =
            p.vis_bits + ((size_t)b * p.Q + (DDT_GUARD(qi < p.Q, 203, p.status + b) ? qi : 0)) * W;
        vis0 = vb[0];
        if (W > 1) vis1 = vb[1];
      }
      // Q row r -> TMEM columns [0,288) as bf16 pairs, from the TMA-staged
      // tile (chunk c: 128 rows x 128 B, 16-byte units swizzled by row & 7).
      // Rows past the sequence hold the next sequence's queries (or zeros
      // past the batch); their results are never written.
      const bool q_ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q_FULL), 0));
      if (q_ok) {
        const unsigned char* qrow = smem + S_RING + r * 128;
#pragma unroll 1
        for (int c = 0; c < kChunksPerTile; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 x = *reinterpret_cast<const uint4*>(qrow + c * (kBM * 128) +
                                                             ((q ^ (r & 7)) << 4));
            v[4 * q + 0] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
          }
          tmem_st32(t_lane + kTmemQ + 32 * c, v);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();  // the ring is refilled by TMA after this
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_Q_TMEM));
      if (!row_barrier_and(q_ok)) failed = true;  // the four row warps agree
      const uint32_t msg_peer0 = map_peer(sbase + O_MSG, peer);
      const uint32_t pfull_peer0 = map_peer(bar(B_P_FULL), peer);

      const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
      float m_run = -INFINITY, l_run = 0.f;
      // One named barrier per tile (before the copy of P): each warp's waits
      // are bounded and their results are AND-ed there, so that all four
      // leave together when one gives up.
      int rj = rot;  // tile_of(jj) without a division
      for (int jj = 0; jj < nt && !failed; ++jj) {
        const int sb = jj & 1;
        const long long t0 = (long long)(jj < nrot ? j_begin + rj : j_begin + jj) * kBN;
        if (jj < nrot && ++rj == nrot) rj = 0;
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_S_FULL + sb), (jj >> 1) & 1));
        tc_fence_after();
        float x[64];  // raw scores q.k (the scale is applied inside the exponent)
        {
          uint32_t sa[32], sc[32];
          tmem_ld32(t_lane + kTmemS + sb * kBN, sa);
          tmem_ld32(t_lane + kTmemS + sb * kBN + 32, sc);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            x[k] = __uint_as_float(sa[k]);
            x[32 + k] = __uint_as_float(sc[k]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));

        // mask: keys past the prefix are visible only along the ancestor path
        if (t0 + kBN > L && !vis_ready) {
          ok = ok && __all_sync(0xffffffffu, mbar_wait(bar(B_TREE), 0));
          if (row_ok) {
            const unsigned long long* vw =
                reinterpret_cast<const unsigned long long*>(smem + S_VIS) + qi * kMaxW;
            vis0 = vw[0];
            vis1 = vw[1];
          }
          vis_ready = true;
        }
        if (t0 + kBN > L) {
          // visibility of the tile's 64 keys as one word: key k is slot t0 + k;
          // slots below L are prefix, slot L + t is tree slot t (bit t of the
          // row's ancestor words vis1:vis0), slots from n_keys on do not exist
          const int np = (int)max(0ll, L - t0);           // prefix keys in the tile, < 64
          const int off = (int)(t0 - L);                 // tree slot of key 0, in (-64, 128)
          const int nk = (int)min(64ll, n_keys - t0);    // keys that exist, in (0, 64]
          unsigned long long tm;
          if (off < 0) tm = vis0 << (-off);
          else if (off == 0) tm = vis0;
          else if (off < 64) tm = (vis0 >> off) | (vis1 << (64 - off));
          else tm = vis1 >> (off - 64);
          const unsigned long long pm = (1ull << np) - 1ull;
          const unsigned long long km = nk >= 64 ? ~0ull : (1ull << nk) - 1ull;
          const unsigned long long m = (pm | tm) & km;
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (!((m >> k) & 1ull)) x[k] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx8[q] = x[q];
#pragma unroll
        for (int k = 8; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], x[k]);
        // the scale is positive, so it commutes with the max
        const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                         p.scale_log2;
        // lazy rescale: the reference max moves only when the row max passes it
        // by 8 (a factor 2^8); O on the peer is then multiplied by `factor`
        float factor = 1.f;
        bool rescale = false;
        if (mt > m_run + 8.f) {
          factor = ex2(m_run - mt);  // 0 when m_run is -inf
          l_run *= factor;
          rescale = jj > 0;
          m_run = mt;
        }
        uint32_t pk[32];
        // p = 2^(x * scale*log2(e) - m); every x is -inf while m is -inf: p = 0
        const float nm = m_run == -INFINITY ? 0.f : -m_run;
        const float2 neg_m = make_float2(nm, nm);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 e = ffma2(make_float2(x[2 * k], x[2 * k + 1]), sl2, neg_m);
          const float2 pp = make_float2(ex2(e.x), ex2(e.y));
          pk[k] = pack_bf16(pp.x, pp.y);
          acc[k & 3] = fadd2(acc[k & 3], pp);
        }
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        const float2 a = fadd2(a01, a23);
        l_run += a.x + a.y;

        // outgoing message slot jj % kMsgSlots (and the peer's) is free once
        // the peer has finished PV of the tile that used it before
        const int mb = jj % kMsgSlots;
        ok = ok && (jj < kMsgSlots ||
                    __all_sync(0xffffffffu, mbar_wait_cluster(bar(B_P_FREE + mb),
                                                              ((jj / kMsgSlots) - 1) & 1)));
        unsigned char* msg = smem + S_STAGE + mb * kMsgStride;
        const uint32_t msg_s = sbase + S_STAGE + mb * kMsgStride;
        const uint32_t p_row = msg_s + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = p_row + ((uint32_t)(c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                       "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
        reinterpret_cast<float*>(msg + kPBytes)[r] = rescale ? factor : 1.f;
        const bool any_rescale = __any_sync(0xffffffffu, rescale);
        if (lane == 0) reinterpret_cast<uint32_t*>(msg + kPBytes + kBM * 4)[qd] = any_rescale;
        fence_proxy_async_smem();
        if (!row_barrier_and(ok)) {
          failed = true;
          break;
        }
        if (tid == 64)
          bulk_copy_to_peer(msg_peer0 + mb * kMsgStride, msg_s, kMsgBytes, pfull_peer0 + 8 * mb);
      }

      // ---- finish: lse here, 1/l to the peer --------------------------------
      if (!failed) {
        const bool live = l_run > 0.f;
        const long long grow = row0 + r;
        if (row_ok) {
          const float lse_v =
              live ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
          if (p.n_split == 1) {
            if (p.lse && DDT_GUARD(grow < total_rows, 204, p.status + b)) p.lse[grow] = lse_v;
          } else {
            p.part_lse[(long long)sp * total_rows + grow] = lse_v;
          }
        }
        reinterpret_cast<float*>(smem + S_FIN)[r] = live ? 1.f / l_run : 0.f;
        fence_proxy_async_smem();
      }
      row_barrier();
      if (tid == 64 && !failed)
        bulk_copy_to_peer(map_peer(sbase + O_FIN, peer), sbase + S_FIN, kFinBytes,
                          map_peer(bar(B_FIN_FULL), peer));
    }
  } else {
    // ========================= O-CTA =========================
    if (warp == 0) {
      int u = 0;
      if (lane == 0) {  // TMA: one 64 KB request (the c_kv part) per tile
        prefetch_tmap(&tm_o);
        for (; u < nt; ++u) {
          const int slot = u % kStages;
          if (u >= kStages && !mbar_wait(bar(B_HALF_EMPTY + slot), ((u / kStages) - 1) & 1)) {
            failed = true;
            break;
          }
          mbar_expect_tx(bar(B_HALF_FULL + slot), kTileO);
          tma_load_3d(sbase + O_RING + slot * kTileO, &tm_o, 0, (int)krow_of(u), 0,
                      bar(B_HALF_FULL + slot));
        }
        for (int v = max(0, u - kStages); v < u; ++v)
          if (!mbar_wait(bar(B_HALF_FULL + v % kStages), (v / kStages) & 1)) failed = true;
      }
      // keys past the end of the sequence in the last tile: the warp zeroes
      // their values so that 0 * (whatever the page holds) cannot turn into NaN
      if (__shfl_sync(0xffffffffu, (!failed && u == nt) ? 1 : 0, 0)) {
        const long long t0 = (long long)(j_begin + nt - 1) * kBN;
        if (t0 + kBN > n_keys) {
          unsigned char* base = smem + O_RING + ((nt - 1) % kStages) * kTileO;
          const int r0 = (int)(n_keys - t0);
          for (int e = lane; e < (kBN - r0) * 64; e += 32) {  // 16-byte units
            const int rr = r0 + (e >> 6), c = (e >> 3) & 7, q = e & 7;
            reinterpret_cast<uint4*>(base + c * kChunkBytes + (rr >> 3) * 1024 +
                                     (rr & 7) * 128)[q] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TAIL_OK));
      }
    } else if (warp == 1) {
      if (lane == 0) {  // PV: A = P (K-major, from the S-CTA), B = V half (MN-major)
        int n_flag = 0;
        for (int jj = 0; jj < nt && !failed; ++jj) {
          const int mb = jj % kMsgSlots;
          if (!mbar_wait_cluster(bar(B_P_FULL + mb), (jj / kMsgSlots) & 1)) {
            failed = true;
            break;
          }
          const unsigned char* msg = smem + O_MSG + mb * kMsgStride;
          const uint4 fl = *reinterpret_cast<const uint4*>(msg + kPBytes + kBM * 4);
          if (jj > 0 && (fl.x | fl.y | fl.z | fl.w)) {  // row warps rescale O first
            if (!mbar_wait(bar(B_O_READY), n_flag & 1)) {
              failed = true;
              break;
            }
            ++n_flag;
          }
          const int slot = jj % kStages;
          if (!mbar_wait(bar(B_HALF_FULL + slot), (jj / kStages) & 1) ||
              (jj == nt - 1 && !mbar_wait(bar(B_TAIL_OK), 0))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t pa = sbase + O_MSG + mb * kMsgStride;
          const uint32_t h0 = sbase + O_RING + slot * kTileO;
          const uint32_t h1 = h0 + kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t ad = smem_desc(pa + kk * 32, 16, 1024, kSwizzle128B);
            const uint32_t acc = (jj > 0 || kk > 0) ? 1u : 0u;
            umma_bf16(tmem, ad, smem_desc(h0 + kk * 2048, kChunkBytes, 1024, kSwizzle128B),
                      kIdescPV, acc);
            umma_bf16(tmem + 256, ad,
                      smem_desc(h1 + kk * 2048, kChunkBytes, 1024, kSwizzle128B), kIdescPV, acc);
          }
          umma_commit(bar(B_PV_DONE + mb));
          umma_commit(bar(B_HALF_EMPTY + slot));
        }
        umma_commit(bar(B_MMA_DONE));
        if (!mbar_wait(bar(B_MMA_DONE), 0)) failed = true;
      }
    } else if (warp >= 2 && warp <= 5) {
      // ---------------- row warps: rescales, message slot recycling, output ---
      const int qd = warp & 3;
      const int r = qd * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
      const int lr = rt * kBM + r;
      const bool row_ok = lr < QH;
      const uint32_t pfree_peer0 = map_peer(bar(B_P_FREE), peer);
      for (int jj = 0; jj < nt; ++jj) {
        const int mb = jj % kMsgSlots;
        bool ok = __all_sync(0xffffffffu,
                             mbar_wait_cluster(bar(B_P_FULL + mb), (jj / kMsgSlots) & 1));
        if (!row_barrier_and(ok)) {
          failed = true;
          break;
        }
        const unsigned char* msg = smem + O_MSG + mb * kMsgStride;
        const uint4 fl = *reinterpret_cast<const uint4*>(msg + kPBytes + kBM * 4);
        if (jj > 0 && (fl.x | fl.y | fl.z | fl.w)) {
          // only the quadrants whose flag is set touch their O rows
          const uint32_t mine = qd == 0 ? fl.x : qd == 1 ? fl.y : qd == 2 ? fl.z : fl.w;
          const float f = reinterpret_cast<const float*>(msg + kPBytes)[r];
          ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PV_DONE + (jj - 1) % kMsgSlots),
                                                 ((jj - 1) / kMsgSlots) & 1));
          if (!row_barrier_and(ok)) {
            failed = true;
            break;
          }
          if (mine) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 16; ++c) {
              uint32_t ov[32];
              tmem_ld32(t_lane + 32 * c, ov);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * f);
              tmem_st32(t_lane + 32 * c, ov);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_O_READY));
        }
        // slot mb is free once PV of tile jj has completed; all row warps move
        // on together so that no warp can fall a message behind
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PV_DONE + mb), (jj / kMsgSlots) & 1));
        if (!row_barrier_and(ok)) {
          failed = true;
          break;
        }
        if (tid == 64) {
          if (jj + kMsgSlots < nt) mbar_expect_tx(bar(B_P_FULL + mb), kMsgBytes);
          mbar_arrive_cluster_relaxed(pfree_peer0 + 8 * mb);
        }
      }
      // ---- epilogue: O / l ---------------------------------------------------
      if (!__all_sync(0xffffffffu, !failed && mbar_wait_cluster(bar(B_FIN_FULL), 0) &&
                                       mbar_wait(bar(B_PV_DONE + (nt - 1) % kMsgSlots),
                                                 ((nt - 1) / kMsgSlots) & 1)))
        failed = true;
      if (!failed) {
        // Each row (512 bf16: the output, or this unit's split-KV partial) is
        // staged in shared memory (the ring and message slots are idle once the
        // last PV has completed) and written with one 1 KB bulk copy: a warp's
        // direct stores would touch 32 rows 1 KB apart.
        tc_fence_after();
        const float inv_l = reinterpret_cast<const float*>(smem + O_FIN)[r];
        const long long grow = row0 + r;
        unsigned char* stage = smem + O_RING + r * kOutStride;
        const uint32_t stage_s = sbase + O_RING + r * kOutStride;
#pragma unroll 1
        for (int c = 0; c < 16; c += 2) {  // two 32-column groups per wait
          uint32_t ov[2][32];
          tmem_ld32(t_lane + 32 * c, ov[0]);
          tmem_ld32(t_lane + 32 * (c + 1), ov[1]);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint4* dst = reinterpret_cast<uint4*>(stage + (c + h) * 64);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16(__uint_as_float(ov[h][8 * q + 0]) * inv_l,
                                            __uint_as_float(ov[h][8 * q + 1]) * inv_l),
                                  pack_bf16(__uint_as_float(ov[h][8 * q + 2]) * inv_l,
                                            __uint_as_float(ov[h][8 * q + 3]) * inv_l),
                                  pack_bf16(__uint_as_float(ov[h][8 * q + 4]) * inv_l,
                                            __uint_as_float(ov[h][8 * q + 5]) * inv_l),
                                  pack_bf16(__uint_as_float(ov[h][8 * q + 6]) * inv_l,
                                            __uint_as_float(ov[h][8 * q + 7]) * inv_l));
          }
        }
        fence_proxy_async_smem();
        if (row_ok && DDT_GUARD(grow < total_rows, 205, p.status + b))
          bulk_s2g(p.n_split == 1 ? p.out + grow * kC
                                  : p.part_o + ((long long)sp * total_rows + grow) * kC,
                   stage_s, 1024);
        bulk_commit();
        bulk_wait0();
      }
    } else if (warp == 6) {
      // ---------------- the fused tree build --------------------------------
      if (builds) {
        bool bad = false;
        const int n = fused_build(p.tf, b, smem + O_BUILD, &bad);
        // the S-CTA needs the ancestor words first; the outputs follow
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          bulk_copy_to_peer(map_peer(sbase + S_VIS, peer),
                            sbase + O_BUILD + (uint32_t)offsetof(tb::Smem, anc), vis_bytes,
                            map_peer(bar(B_TREE), peer));
        if (designated) fused_write(p, b, smem + O_BUILD, n, bad);
      }
    }
  }

  // the ancestor words sent by the peer have landed before this CTA leaves
  if (builds && rank == 0 && tid == 0 && !mbar_wait(bar(B_TREE), 0)) failed = true;
  if (failed) atomicOr(p.status + b, DDT_ST_TIMEOUT);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // every copy and remote arrive between the two CTAs has landed
}

// Merge of the split-KV partials: o = sum_s w_s o_s / sum_s w_s with
// w_s = exp(lse_s - max lse); one warp per query row, 16 columns per lane.
// The partials are bf16 (each already normalised by its own sum), which
// halves their round trip through memory; the merge runs in fp32.
__device__ void combine_row(long long row, long long total_rows, int n_split,
                            const __nv_bfloat16* __restrict__ part_o,
                            const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out,
                            float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
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
      const uint4* src =
          reinterpret_cast<const uint4*>(part_o + ((long long)s * total_rows + row) * kC) +
          lane * 2;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 v = src[q];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
          acc[8 * q + 2 * e] = fmaf(w, f.x, acc[8 * q + 2 * e]);
          acc[8 * q + 2 * e + 1] = fmaf(w, f.y, acc[8 * q + 2 * e + 1]);
        }
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

__device__ void combine_row_wide(long long row, long long total_rows, int n_split,
                            const __nv_bfloat16* __restrict__ part_o,
                            const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out,
                            float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  // Eight partials at a time: their lse and this lane's 16 dims are all
  // requested before any is used, so a row of many partials waits for one
  // memory round trip per eight of them, not two per partial.
  constexpr int kBatch = 8;
  float m = -INFINITY;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  for (int s0 = 0; s0 < n_split; s0 += kBatch) {
    float ls[kBatch];
    uint4 v[kBatch][2];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int s = s0 + j;
      if (s < n_split) {
        ls[j] = part_lse[(long long)s * total_rows + row];
        const uint4* src =
            reinterpret_cast<const uint4*>(part_o + ((long long)s * total_rows + row) * kC) +
            lane * 2;
        v[j][0] = src[0];
        v[j][1] = src[1];
      } else {
        ls[j] = -INFINITY;
      }
    }
    // the running reference max moves to the batch's max; earlier sums rescale
    float mb = m;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) mb = fmaxf(mb, ls[j]);
    if (mb == -INFINITY) continue;
    if (mb != m) {
      const float r = m == -INFINITY ? 0.f : expf(m - mb);
      wsum *= r;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] *= r;
      m = mb;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (ls[j] == -INFINITY) continue;
      const float w = expf(ls[j] - m);
      wsum += w;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t wv[4] = {v[j][q].x, v[j][q].y, v[j][q].z, v[j][q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
          acc[8 * q + 2 * e] = fmaf(w, f.x, acc[8 * q + 2 * e]);
          acc[8 * q + 2 * e + 1] = fmaf(w, f.y, acc[8 * q + 2 * e + 1]);
        }
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

// Split-KV merge: one warp per query row. Launched as the programmatic
// dependent of the step's accept + compaction kernel, it runs beside it and
// then waits for it before exiting, so work queued after the merge still
// finds the step complete (without such a predecessor the wait returns at
// once). kWide takes partials eight at a time: faster from five partials up
// when the rows are few (the q_len 1 steps split over tens of key ranges,
// where each row's chain of memory round trips is the whole merge); with two
// partials, or with enough rows for several blocks per SM, the one-at-a-time
// loop wins, its 48 registers against about 200 keeping more warps resident.
constexpr int kCombineWideFrom = 5;
constexpr long long kCombineWideRows = 8LL * 152 * 4;
template <bool kWide>
__global__ void __launch_bounds__(256) k_combine(long long total_rows, int n_split,
                                                 const __nv_bfloat16* __restrict__ part_o,
                                                 const float* __restrict__ part_lse,
                                                 __nv_bfloat16* __restrict__ out,
                                                 float* __restrict__ lse_out) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row < total_rows) {
    if (kWide) combine_row_wide(row, total_rows, n_split, part_o, part_lse, out, lse_out);
    else combine_row(row, total_rows, n_split, part_o, part_lse, out, lse_out);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- host side

int sm_count() {
  static int cached[64] = {};
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return n;
  if (cached[dev] == 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    cached[dev] = n;
  return cached[dev] ? cached[dev] : n;
}

// One way of running a launch: the row-tile height (128: two-CTA clusters,
// this file; 256: four-CTA clusters on paired SMs, verify_attn_pair.cu), the
// number of key ranges each sequence is split into, and the modelled cost.
struct Plan {
  int rows;     // 128 or 256
  int n_rt, n_split;
  long long units;
  double cost;  // in key-tile times of the 128-row kernel
};

// Cost model of a launch, in SM cycles, from cycle traces of both kernels on
// GB300: a unit (one cluster's rows x key range) costs a fixed start (Q load,
// instruction fetch, the first tiles through the pipeline, the epilogue) plus
// its key tiles. The 128-row kernel runs its units in waves of `per_wave`
// clusters, each paying the whole start; the 256-row kernel keeps `per_wave`
// clusters resident, each walking its list of units, and a unit that follows
// another in the same cluster pays only the part of the start that does not
// overlap the previous unit's end (`unit_next`). A split key range adds the
// merge pass, which streams every partial once at HBM speed.
struct KernelCost {
  int rows;           // query rows per tile
  int keys_per_tile;  // keys per step of the key walk
  double unit_start;  // cycles
  double unit_next;   // cycles, for a unit after another in the same cluster
  double per_64_keys; // cycles per 64 keys of one unit
};
constexpr KernelCost kCost128 = {128, 64, 45000.0, 45000.0, 2400.0};
constexpr KernelCost kCost256 = {256, 128, 40000.0, 12000.0, 1750.0};
constexpr double kMergeBytesPerCycle = 3200.0;  // about 6.6 TB/s at 2.07 GHz

Plan make_plan(const ddt_attn_dims& d, const KernelCost& k, long long per_wave) {
  Plan pl;
  pl.rows = k.rows;
  const long long QH = (long long)d.Q * d.H;
  pl.n_rt = (int)((QH + k.rows - 1) / k.rows);
  const long long base = (long long)d.B * pl.n_rt;
  const long long max_len = d.max_len > d.Q ? d.max_len : d.Q;
  const long long n_tiles = (max_len + k.keys_per_tile - 1) / k.keys_per_tile;
  const double rows_total = (double)d.B * (double)QH;
  if (per_wave < 1) per_wave = 1;
  pl.cost = 1e300;
  pl.n_split = 1;
  for (long long s = 1; s <= 64 && s <= n_tiles; ++s) {
    const long long units = base * s;
    const double waves = (double)((units + per_wave - 1) / per_wave);
    // tiles of the longest unit (the kernels give every unit but the last
    // one tile more than an even share when the range is split)
    const long long tpu = s > 1 ? (n_tiles + s) / s : n_tiles;
    const double work = (double)tpu * (double)(k.keys_per_tile / 64) * k.per_64_keys;
    const double merge =
        s > 1 ? 3000.0 + (double)(s + 1) * rows_total * 1028.0 / kMergeBytesPerCycle : 0.0;
    const double cost = waves * work + k.unit_start + (waves - 1.0) * k.unit_next + merge;
    if (cost < pl.cost - 1e-9) {
      pl.cost = cost;
      pl.n_split = (int)s;
    }
  }
  pl.units = base * pl.n_split;
  return pl;
}

Plan plan_128(const ddt_attn_dims& d) { return make_plan(d, kCost128, sm_count() / 2); }
Plan plan_256(const ddt_attn_dims& d) {
  int per_wave = verify_attn_pair_clusters_per_wave();
  if (per_wave < 1) per_wave = sm_count() / 4;
  return make_plan(d, kCost256, per_wave);
}

// The launch's plan: the cheaper of the two kernels by the cost model. The
// 256-row kernel moves half the bytes per FLOP and runs a key tile faster per
// SM, but pads a sequence's Q*H rows to a multiple of 256 (q_len 65 x 64
// heads: 4160 rows in 4352; q_len 17 x 64 heads: 1088 rows in 1280), which
// the model counts as work. The environment variable DDT_VERIFY_ATTN_ROWS (128 or 256)
// overrides the choice.
Plan choose_plan(const ddt_attn_dims& d) {
  const char* env = getenv("DDT_VERIFY_ATTN_ROWS");
  if (env != nullptr && strcmp(env, "128") == 0) return plan_128(d);
  if (env != nullptr && strcmp(env, "256") == 0) return plan_256(d);
  const Plan p128 = plan_128(d);
  if (verify_attn_pair_clusters_per_wave() <= 0) return p128;
  const Plan p256 = plan_256(d);
  return p256.cost < p128.cost ? p256 : p128;
}

size_t workspace_of(const ddt_attn_dims& d, const Plan& pl) {
  if (pl.n_split <= 1) return 0;
  const size_t rows = (size_t)d.B * d.Q * d.H;
  const size_t bytes = (size_t)pl.n_split * rows * (kC * sizeof(__nv_bfloat16) + sizeof(float));
  return (bytes + 255) & ~size_t(255);
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

bool encode_kv_3d(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_chunks) {
  auto fn = encoder();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, rows, (cuuint64_t)kChunksPerTile};
  cuuint64_t strides[2] = {(cuuint64_t)(kC + kR) * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kBN, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q as {64 dims, rows, 8 chunks} (q_lat, row stride 1 KB) and {64 dims, rows}
// (q_pe, row stride 128 B); a box of 128 rows lands as 128-row x 128-byte
// swizzled chunks, the layout the row warps read back for TMEM.
bool encode_q(CUtensorMap* ml, CUtensorMap* mp, const void* q_lat, const void* q_pe,
              uint64_t rows) {
  auto fn = encoder();
  if (fn == nullptr) return false;
  cuuint64_t dl[3] = {64, rows, (cuuint64_t)(kC / 64)};
  cuuint64_t sl[2] = {(cuuint64_t)kC * 2, 128};
  cuuint32_t bl[3] = {64, (cuuint32_t)kBM, (cuuint32_t)(kC / 64)};
  cuuint32_t e3[3] = {1, 1, 1};
  if (fn(ml, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_lat), dl, sl, bl, e3,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cuuint64_t dp[2] = {64, rows};
  cuuint64_t sp[1] = {(cuuint64_t)kR * 2};
  cuuint32_t bp[2] = {64, (cuuint32_t)kBM};
  cuuint32_t e2[2] = {1, 1};
  return fn(mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_pe), dp, sp, bp, e2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Enough for either tile height, so that the size a caller obtained stays
// valid whichever kernel a launch picks.
size_t verify_attn_bf16_workspace(const ddt_attn_dims& d) {
  const size_t a = workspace_of(d, plan_128(d)), b = workspace_of(d, plan_256(d));
  return a > b ? a : b;
}

cudaError_t launch_verify_attn_bf16(const ddt_attn_dims& d, const void* q_lat, const void* q_pe,
                                    const void* kv, const int32_t* block_table,
                                    const int32_t* prefix_len, const uint64_t* vis_bits,
                                    void* out, float* lse, int32_t* status, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream,
                                    const TreeFuse* fuse, const AcceptCompactArgs* then) {
  const Plan pl = choose_plan(d);
  const long long rows = (long long)d.B * d.Q * d.H;
  if (d.kv_rows < 1 || rows > 0x7fffffffLL || d.kv_rows > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  if (pl.n_split > 1 && (workspace == nullptr || workspace_bytes < workspace_of(d, pl)))
    return cudaErrorInvalidValue;
  __nv_bfloat16* part_o = nullptr;
  float* part_lse = nullptr;
  if (pl.n_split > 1) {
    part_o = static_cast<__nv_bfloat16*>(workspace);
    part_lse = reinterpret_cast<float*>(part_o + (size_t)pl.n_split * rows * kC);
  }
  cudaError_t e;
  if (pl.rows == 256) {
    e = launch_verify_attn_pair(d, pl.n_split, q_lat, q_pe, kv, block_table, prefix_len, vis_bits,
                                out, lse, status, part_o, part_lse, stream, fuse);
  } else {
    // the cache as {64 dims, rows, 9 chunks} with strides (row, 128 B)
    CUtensorMap tm_s, tm_o, tm_ql, tm_qp;
    if (!encode_kv_3d(&tm_s, kv, (uint64_t)d.kv_rows, kChunksPerTile) ||
        !encode_kv_3d(&tm_o, kv, (uint64_t)d.kv_rows, 8) ||
        !encode_q(&tm_ql, &tm_qp, q_lat, q_pe, (uint64_t)rows))
      return cudaErrorInvalidValue;
    Params p;
    p.B = d.B; p.Q = d.Q; p.H = d.H;
    p.page_size = d.page_size; p.max_pages = d.max_pages; p.kv_rows = d.kv_rows;
    p.scale_log2 = d.scale * 1.4426950408889634f;
    p.n_rt = pl.n_rt; p.n_split = pl.n_split;
    p.block_table = block_table; p.prefix_len = prefix_len;
    p.vis_bits = reinterpret_cast<const unsigned long long*>(vis_bits);
    p.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
    p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse; p.status = status;
    p.part_o = part_o; p.part_lse = part_lse;
    p.fuse = fuse != nullptr ? 1 : 0;
    p.tf = fuse != nullptr ? *fuse : TreeFuse{};
    static int smem_set[64] = {};
    e = ensure_smem_limit(k_verify_attn_bf16, (int)kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    k_verify_attn_bf16<<<(unsigned)(pl.units * 2), kThreads, kSmemBytes, stream>>>(
        tm_s, tm_o, tm_ql, tm_qp, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if (pl.n_split == 1) return then != nullptr ? launch_accept_compact(*then, stream) : e;
  const bool wide = pl.n_split >= kCombineWideFrom && rows <= kCombineWideRows;
  if (then == nullptr) {
    if (wide)
      k_combine<true><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
          rows, pl.n_split, part_o, part_lse, static_cast<__nv_bfloat16*>(out), lse);
    else
      k_combine<false><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
          rows, pl.n_split, part_o, part_lse, static_cast<__nv_bfloat16*>(out), lse);
    return cudaGetLastError();
  }
  // accept + compaction first (it needs the tree and the finished cache
  // reads of the attention, not its output), then the merge as its
  // programmatic dependent: k_accept_compact lets dependents start at once,
  // and the merge's inputs come from the attention, which completed before
  // k_accept_compact began, so the two run side by side
  e = launch_accept_compact(*then, stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wide ? k_combine<true> : k_combine<false>, rows, pl.n_split,
                            static_cast<const __nv_bfloat16*>(part_o),
                            static_cast<const float*>(part_lse), static_cast<__nv_bfloat16*>(out),
                            lse);
}

int verify_attn_bf16_rows_per_tile(const ddt_attn_dims& d) { return choose_plan(d).rows; }
int verify_attn_bf16_splits(const ddt_attn_dims& d) { return choose_plan(d).n_split; }

}  // namespace ddt
