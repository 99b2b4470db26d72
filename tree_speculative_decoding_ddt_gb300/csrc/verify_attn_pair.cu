// B. Tree-verify MLA-absorb attention on paired SMs: 256-row tiles, four CTAs
// per cluster, tcgen05 MMAs of M = 256 shared by two SMs (cta_group::2).
//
// "The Checkpoint: Committing a Working Native DDTree Engine", section "The
// Message": verify attention in MLA absorb form, tree [verified_id, drafts]
// at cache positions L + depth, mask [ones over the prefix | visibility];
// "The Milestone Commit", section "Input Knowledge Required": the latent
// cache of Kimi K2.6 (kv_lora_rank 512, plus a 64-wide rope part).
//
// Same arithmetic as the 128-row kernel (verify_attn_bf16.cu): per sequence
// the Q*H query rows (row = query position * H + head) share one latent KV
// head, S = [q_lat | q_pe] . [c_kv | k_pe]^T (contraction 576) and
// O = softmax(S * scale, masked) . c_kv (output 512), online softmax, fp32
// accumulation in TMEM. What changes is how a tile is
// spread over the SMs. A 128 x 512 fp32 O fills the 512 TMEM columns of an
// SM, so S and O still live on different SMs, and each side is now a pair of
// SMs running one M = 256 MMA:
//   * ranks 0, 1 (the S pair) hold Q rows [0,128) and [128,256) of the tile:
//     q_lat in TMEM (256 columns: staged through the key ring by TMA and
//     copied in by the MMA issuer with tcgen05.cp), q_pe in shared memory
//     (16 KB). S is taken
//     over 128-key tiles: each S-CTA loads one 64-key half of the tile (64
//     keys x 576 dims, 72 KB, one TMA request) and the pair MMA (issued by
//     rank 0; N = 128, so 36 MMA instructions per 128 keys) writes S for its
//     128 rows x all 128
//     keys into each CTA's TMEM (two 128-column buffers). Eight softmax warps
//     per CTA take two threads per row, one per 64-key half; each half ships
//     its P block (bf16, 16 KB) plus per-row rescale factors to the O-CTA of
//     the same rows;
//   * ranks 2, 3 (the O pair) hold O rows [0,128) and [128,256) in TMEM and
//     consume the P blocks in key order, 64 keys at a time: each loads HALF of
//     the value dims of the block (64 keys x 256 dims, 32 KB: rank 2 dims
//     [0,128) and [256,384), rank 3 the other two) and the pair MMA (issued
//     by rank 2) accumulates O += P V.
// Against one 128-row tile per SM pair this halves the bytes every CTA stages
// per FLOP and the L2 traffic of the key walk. A single thread issues a
// tcgen05.mma with A in TMEM only about every 70 cycles whatever N is, so the
// S tile is as wide as TMEM allows (N = 128) to keep the MMA count per key low.
//
// Warp roles (352 threads). S-CTAs: warp 0 TMA (its Q rows, then its key
// halves), warp 1 TMEM allocation and then (rank 0) the first MMA issuer or
// (rank 1) the relay that tells rank 0 an S buffer has been read, warps 2-9
// softmax (two groups of four warps taking alternate key tiles; warp w holds
// lane quadrant w % 4), warp 10 (rank 0) the second MMA issuer (the two take
// alternate key tiles, which keeps the tensor pipe busy while one of them is
// issuing) or (rank 1) the relay of its key halves' arrival. O-CTAs: warp 0
// TMA, warp 1 TMEM allocation and (rank 2) the PV issuer, warps 2-5 row warps
// (rescales, output), warp 6 of rank 2 the fused tree build.
//
// Units and clusters. A unit is one (sequence, 256-row tile, key range). The
// grid holds at most as many clusters as are resident at once, and each
// cluster walks a fixed list of units, so that the next unit's start (its
// page checks, the Q load into TMEM, the first key tiles) runs while the
// previous unit's last tiles and epilogue finish: the S side starts unit k+1
// as soon as the MMAs of unit k have read their last key tile, and the O
// side's epilogue of unit k overlaps it. Every barrier keeps its phase count
// across units. Warp 0 of each CTA reads a unit's prefix length, checks its
// pages and publishes them (two buffers, by unit parity) before the other
// roles take the unit.
#include <cuda_bf16.h>
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>

#include <cudaTypedefs.h>

#include "ddt_internal.cuh"
#include "sm100_ptx.cuh"
#include "tree_build_warp.cuh"

namespace ddt {
DDT_CHECKS_FILE(pair)
namespace {

using namespace sm100;

constexpr int kTM = 256;  // query rows per tile
constexpr int kHM = 128;  // query rows per CTA
constexpr int kBK = 64;   // keys per block (one P message, one value stage)
constexpr int kBS = 128;  // keys per S tile (two blocks; one per S-CTA)
constexpr int kC = 512;
constexpr int kR = 64;
constexpr int kThreads = 352;
constexpr int kStagesK = 2;   // S-CTA key stages (one 64-key half of an S tile each)
constexpr int kStagesV = 4;   // O-CTA value stages (one 64-key block each)
constexpr int kStageSlots = 3;  // S-CTA: outgoing P blocks (free once copied)
constexpr int kMsgSlots = 4;    // O-CTA: incoming P blocks (free once PV has read them)

constexpr int kChunks = (kC + kR) / 64;                   // 9 chunks of 64 dims
// Key loads per 64-key half, each released to the producer when its MMAs are
// done. Splitting the half into 3 or 9 loads, so that the next tile's first
// chunks land early, measured slower at c4 (1557 and 1944 us against 1487):
// the per-request cost of the smaller loads outweighs the earlier start.
constexpr int kKGroups = 1;
constexpr int kGroupChunks = kChunks / kKGroups;          // chunks per key load
constexpr uint32_t kKChunk = kBK * 128;                   // 64 keys x 128 B
constexpr uint32_t kTileK = kChunks * kKChunk;            // an S-CTA's key half: 72 KB
constexpr uint32_t kVChunk = kBK * 128;                   // 64 keys x 128 B
constexpr uint32_t kTileV = 4 * kVChunk;                  // an O-CTA's value half: 32 KB
constexpr uint32_t kPBytes = kHM * 128;                   // P: 128 rows x 64 keys bf16
constexpr uint32_t kMsgBytes = kPBytes + kHM * 4 + 16;    // P | per-row factor | 4 warp flags
constexpr uint32_t kMsgStride = 17408;
constexpr uint32_t kFinBytes = kHM * 4;
constexpr uint32_t kQlHalf = kHM * (kC / 2) * 2;          // half the q_lat dims of the rows: 64 KB
constexpr uint32_t kQpBytes = kHM * kR * 2;               // q_pe rows: 16 KB

// S-CTA shared memory
constexpr uint32_t S_RING = 0;
constexpr uint32_t S_QPE = S_RING + kStagesK * kTileK;   // q_pe (SW128, K-major)
constexpr uint32_t S_STAGE = S_QPE + kQpBytes;            // outgoing messages
constexpr uint32_t S_FIN = S_STAGE + kStageSlots * kMsgStride;  // [2][128] 1/l, by unit parity
constexpr uint32_t S_XCH = S_FIN + 2 * kFinBytes;  // running max handoff [128], final (m, l) [2][128][2]
constexpr uint32_t kVisBuf = kMaxQ * kMaxW * 8;
constexpr uint32_t S_VIS = S_XCH + 2048 + 512;  // [2] ancestor words of the fused build, by unit parity
constexpr uint32_t S_END = S_VIS + 2 * kVisBuf;
// O-CTA shared memory
constexpr uint32_t O_RING = 0;
constexpr uint32_t O_OUT = O_RING + 2 * kTileV;  // output staging in value stage 2: [warp][2][32 x 128 B]
constexpr uint32_t kOutBox = 32 * 128;           // 32 rows x 64 dims bf16, one TMA store
constexpr uint32_t O_MSG = O_RING + kStagesV * kTileV;
constexpr uint32_t O_FIN = O_MSG + kMsgSlots * kMsgStride;  // [2][128] 1/l, by unit parity
constexpr uint32_t O_GO = O_FIN + 2 * kFinBytes;  // message index of the current GO call (-1: the end)
constexpr uint32_t O_PEERFLAG = O_GO + 256;       // rank 2: rank 3's rescale flags [slot][16 B]
constexpr uint32_t O_BUILD = O_GO + 1024;
constexpr uint32_t kBuildBytes = (uint32_t)tb::smem_bytes(kFuseMaxCand, 1);
constexpr uint32_t O_END = O_BUILD + ((kBuildBytes + 1023) & ~1023u);

// Sequences per launch up to which the clusters take them longest first.
constexpr int kLongestFirstMax = 352;
constexpr int kBtMax = 512;  // page indices of a unit kept in shared memory
constexpr uint32_t OFF_BT = (S_END > O_END ? S_END : O_END);  // [2][kBtMax], by unit parity
constexpr uint32_t OFF_ORDER = OFF_BT + 2 * kBtMax * 4;      // [kLongestFirstMax]: sequence of rank i
constexpr uint32_t OFF_INFO = OFF_ORDER + kLongestFirstMax * 4;  // [2] UnitInfo, by unit parity
constexpr uint32_t OFF_CNT = OFF_INFO + 128;  // softmax warps' unit counters [8 warps][8]
constexpr uint32_t OFF_BAR = OFF_CNT + 8 * 32;
constexpr uint32_t kSmemBytes = OFF_BAR + 1024 + 1024;
static_assert(kQlHalf <= kTileK, "each half of q_lat is staged in one stage of the key ring");
static_assert(S_STAGE % 1024 == 0 && O_MSG % 1024 == 0 && kMsgStride % 1024 == 0, "alignment");
static_assert(kMsgBytes <= kMsgStride && kMsgBytes % 16 == 0, "message size");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(O_OUT % 1024 == 0 && O_OUT + 4 * 2 * kOutBox <= O_RING + 3 * kTileV,
              "the output is staged in value stage 2");
static_assert(4 * 8 * kOutBox <= kStagesV * kTileV,
              "a cluster's last unit stages all its output boxes in the value ring");
static_assert(S_QPE % 1024 == 0, "q_pe is an MMA operand");
static_assert(S_VIS % 16 == 0 && kVisBuf % 16 == 0, "ancestor words are bulk-copied");
static_assert(offsetof(tb::Smem, anc) % 16 == 0, "ancestor words are bulk-copied");
static_assert(kLongestFirstMax <= kThreads, "one thread per sequence ranks the lengths");

enum Bar {
  // S-CTAs
  // key ring barriers are per chunk group of a stage: index stage * kKGroups + group
  B_RING_FULL = 0,                                   // this CTA's group landed
  B_RING_PEER = B_RING_FULL + kStagesK * kKGroups,   // rank 0: rank 1's group landed (relay)
  B_RING_EMPTY = B_RING_PEER + kStagesK * kKGroups,  // both: the MMAs of the group are done
  B_S_FULL = B_RING_EMPTY + kStagesK * kKGroups,     // +buffer; both (pair MMA commit)
  B_S_EMPTY = B_S_FULL + 2,               // +buffer; rank 0: its 4 warps of one group + rank 1's relay
  B_S_READ = B_S_EMPTY + 2,               // +buffer; rank 1: its 4 warps of one group read S
  B_Q_FULL = B_S_READ + 2,                // +half; q_lat dims [256h, 256h + 256) landed (h = 0: and q_pe)
  B_Q_PEER = B_Q_FULL + 2,                // rank 0: both of rank 1's q_lat halves landed (relay)
  B_Q_LOCAL = B_Q_PEER + 1,               // +half; both: the half has been copied into TMEM (pair commit)
  B_Q_TMEM = B_Q_LOCAL + 2,               // rank 0: all q_lat of both CTAs in TMEM (commit)
  B_P_FREE = B_Q_TMEM + 1,                // +O-CTA slot; both (PV commit from rank 2)
  B_STAGE_FREE = B_P_FREE + kMsgSlots,    // +staging slot; the O-CTA saw the copy land
  B_TREE = B_STAGE_FREE + kStageSlots,    // +buffer; ancestor words of the fused build landed
  B_FIN_FREE = B_TREE + 2,                // +buffer; the O-CTA has read the unit's 1/l (4 row warps)
  // O-CTAs
  B_HALF_FULL = B_FIN_FREE + 2,           // +stage; this CTA's value half landed
  B_HALF_PEER = B_HALF_FULL + kStagesV,   // +stage; rank 2: rank 3's value half landed (relay)
  B_HALF_EMPTY = B_HALF_PEER + kStagesV,  // +stage; both (PV commit)
  B_P_FULL = B_HALF_EMPTY + kStagesV,     // +slot; completed by the S-CTA's copy
  B_P_PEER = B_P_FULL + kMsgSlots,        // +slot; rank 2: rank 3's message landed (its flags, 16 B)
  B_PV_DONE = B_P_PEER + kMsgSlots,       // +slot; both (PV commit)
  B_GO = B_PV_DONE + kMsgSlots,           // both: the PV issuer calls the row warps (a rescale, or the end)
  B_O_READY = B_GO + 1,                   // rank 2: +0 its row warps, +1 rank 3's, rescale done
  B_FIN_FULL = B_O_READY + 2,             // +buffer; the unit's 1/l landed
  B_TAIL_OK = B_FIN_FULL + 2,             // rank 2, +buffer: both halves of the unit's last block zeroed
  B_EPI_DONE = B_TAIL_OK + 2,             // rank 2, +buffer: both CTAs' row warps have read O of the unit
  B_OUT_FREE = B_EPI_DONE + 2,            // the output staging has been read (4 row warps)
  // both sides
  B_INFO = B_OUT_FREE + 1,                // +buffer; warp 0 has published the unit's checks
  B_INFO_FREE = B_INFO + 2,               // +buffer; every other role is done with the unit
  B_MMA_DONE = B_INFO_FREE + 2,
  N_BARS = B_MMA_DONE + 1
};
static_assert(N_BARS * 8 + 16 <= 1024, "barrier area");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;    // S-CTA: q_lat [0,256)
constexpr uint32_t kTmemS = 256;  // S-CTA: S buffers [256,384), [384,512)

constexpr uint32_t kIdescS = idesc_bf16_f32(kTM, kBS, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kTM, 256, true);
constexpr uint16_t kMaskS = 0x3;  // ranks 0, 1
constexpr uint16_t kMaskO = 0xC;  // ranks 2, 3

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
  __nv_bfloat16* part_o;
  float* part_lse;
  int fuse;
  int longest_first;  // clusters take the sequences in order of decreasing prefix length
  TreeFuse tf;
};

// What warp 0 of a CTA publishes about a unit.
struct UnitInfo {
  int b, rt, sp;
  int code;     // DDT_ST_CAPACITY / DDT_ST_RANGE, or 0
  long long L;  // prefix length
  int pad[2];
};
static_assert(sizeof(UnitInfo) == 32 && offsetof(UnitInfo, L) == 16 && OFF_INFO % 32 == 0,
              "unit info layout (read by 16- and 8-byte shared loads)");

// Everything else about a unit, derived from its info in the same way by
// every role.
struct Unit {
  long long L, n_keys;
  int b, rt, sp, code;
  int n_blocks;    // 64-key blocks of the sequence
  int j_begin;     // first 128-key tile of the unit's key range
  int nt;          // 128-key tiles of the unit (0: nothing to attend)
  int n_msgs;      // 64-key P blocks of the unit
  int nrot, rot;   // tiles wholly inside the prefix, and where their walk starts
  bool designated; // writes the tree outputs when the build is fused
  bool builds;     // walks tree tiles and so builds the tree when it is fused
};

__device__ __forceinline__ Unit derive_unit(const Params& p, const UnitInfo& ui) {
  Unit u;
  u.L = ui.L; u.b = ui.b; u.rt = ui.rt; u.sp = ui.sp; u.code = ui.code;
  u.n_keys = u.L + p.Q;
  const int n_tiles = (int)((u.n_keys + kBS - 1) / kBS);  // 128-key S tiles
  u.n_blocks = (int)((u.n_keys + kBK - 1) / kBK);          // 64-key blocks
  // the last unit of a split sequence also walks the tree tiles (and builds
  // the tree): the earlier units take the extra tile when the range divides
  const int tps = p.n_split > 1 ? (n_tiles + p.n_split) / p.n_split : n_tiles;
  u.j_begin = u.sp * tps;
  u.nt = u.code ? 0 : max(0, min(n_tiles, u.j_begin + tps) - u.j_begin);
  const int sp_last = u.code ? 0 : (n_tiles - 1) / tps;
  u.designated = p.fuse && u.rt == 0 && u.sp == sp_last;
  // The sequence's last S tile may hold one 64-key block only; its second
  // half is then a phantom: loaded from the first half's rows, fully masked,
  // never sent. Message m of the unit is block 2 * tile_of(m / 2) + m % 2.
  const bool phantom = u.nt > 0 && u.j_begin + u.nt == n_tiles && 2 * n_tiles > u.n_blocks;
  u.n_msgs = 2 * u.nt - (phantom ? 1 : 0);
  // Key walk: tiles wholly inside the prefix from a staggered starting point,
  // the tiles holding tree keys last, in order. Row tiles of a sequence start
  // their walks up to three tiles apart: close enough that the tiles one row
  // tile reads are still in L2 for the others (spreading the starts over the
  // whole prefix cost 2.4x the cache's DRAM bytes once several long sequences
  // were in flight), far enough that they do not all ask for the same lines
  // at the start.
  const int n_pure = (int)(u.L / kBS);
  u.nrot = max(0, min(u.j_begin + u.nt, n_pure) - u.j_begin);
  u.builds = p.fuse && u.nt > u.nrot;
  u.rot = u.nrot > 0 ? (u.rt % 4) % u.nrot : 0;
  return u;
}
// The unit's info as published in shared memory (read with shared loads from
// a 32-bit address, so that no role holds a generic pointer to it).
__device__ __forceinline__ UnitInfo load_info(uint32_t a) {
  UnitInfo ui;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(ui.b), "=r"(ui.rt), "=r"(ui.sp), "=r"(ui.code)
               : "r"(a)
               : "memory");
  uint32_t lo, hi;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(a + 16) : "memory");
  ui.L = (long long)(((unsigned long long)hi << 32) | lo);
  return ui;
}

__device__ __forceinline__ int tile_of(const Unit& u, int jj) {
  return (jj < u.nrot) ? u.j_begin + (jj + u.rot) % u.nrot : u.j_begin + jj;
}
__device__ __forceinline__ int msg_block(const Unit& u, int m) {
  return 2 * tile_of(u, m >> 1) + (m & 1);
}
// cache row of the first key of 64-key block `blk` of the unit's sequence
__device__ __forceinline__ long long block_row(const Params& p, const Unit& u, const int32_t* s_bt,
                                               int blk) {
  const long long t0 = (long long)blk * kBK;
  const long long pi = t0 / p.page_size;
  if (!DDT_GUARD(pi >= 0 && pi < p.max_pages, 101, p.status + u.b)) return 0;
  const int32_t pg = pi < kBtMax ? s_bt[pi] : p.block_table[(size_t)u.b * p.max_pages + pi];
  const long long row = (long long)pg * p.page_size + t0 % p.page_size;
  // a 64-key block must lie inside the cache (the TMA is clamped to row 0 otherwise)
  return DDT_GUARD(row >= 0 && row + kBK <= p.kv_rows, 102, p.status + u.b) ? row : 0;
}

// Unit i of cluster c among G clusters: units are numbered longest first
// (sequence rank, then row tile, then key range); round i hands units
// [iG, iG + G) to the clusters, forwards on even rounds and backwards on odd
// ones, so that a cluster that took a long unit in one round takes a short
// one in the next.
__device__ __forceinline__ long long unit_id(int c, int G, int i) {
  return (long long)i * G + ((i & 1) ? G - 1 - c : c);
}
__device__ __forceinline__ void unit_coords(const Params& p, const int32_t* order, long long uid,
                                            int* b, int* rt, int* sp) {
  *sp = (int)(uid % p.n_split);
  *rt = (int)((uid / p.n_split) % p.n_rt);
  const int rank = (int)(uid / ((long long)p.n_split * p.n_rt));
  *b = p.longest_first ? order[rank] : rank;
}

// Warp 0 of a CTA: the unit's prefix length, capacity and page checks, its
// first kBtMax page indices into shared memory. Identical decision in all four
// CTAs of the cluster (they read the same words).
__device__ void unit_checks(const Params& p, int b, int rt, int sp, int32_t* s_bt, UnitInfo* info,
                            int lane) {
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
  // the first pages are read with the prefix length (the page count depends on it)
  const int32_t pg_first = lane < p.max_pages ? bt[lane] : 0;
  const long long L = p.prefix_len[b];
  const long long n_keys = L + p.Q;
  int code = 0;
  if (L < 0 || n_keys > (long long)p.max_pages * p.page_size || n_keys > 0x7fffffffLL)
    code = DDT_ST_CAPACITY;
  if (code == 0) {
    const long long n_pages = (n_keys + p.page_size - 1) / p.page_size;
    const long long kv_pages = p.kv_rows / p.page_size;
    bool badp = false;
    for (long long q0 = 0; q0 < n_pages; q0 += 8 * 32) {
      int32_t v[8];  // eight loads in flight per lane
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const long long q = q0 + k * 32 + lane;
        v[k] = q == lane ? pg_first : (q < n_pages ? bt[q] : 0);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const long long q = q0 + k * 32 + lane;
        if (q < n_pages) {
          if (q < kBtMax) s_bt[q] = v[k];
          if (v[k] < 0 || v[k] >= kv_pages) badp = true;
        }
      }
    }
    if (__any_sync(0xffffffffu, badp)) code = DDT_ST_RANGE;
  }
  if (lane == 0) {
    info->L = L;
    info->b = b;
    info->rt = rt;
    info->sp = sp;
    info->code = code;
  }
  __threadfence_block();
  __syncwarp();
}

__device__ __forceinline__ int lds_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_s32(uint32_t a, int v) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long lds_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_u64(uint32_t a, unsigned long long v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32x2(uint32_t a, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
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
// named barrier 1 over `n` threads, returning the AND of `ok` over them
__device__ __forceinline__ bool bar1_and(bool ok, uint32_t n) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(n)
      : "memory");
  return r != 0;
}
// named barrier `id` over `n` threads, returning the AND of `ok` over them
__device__ __forceinline__ bool bar1_and_id(bool ok, uint32_t id, uint32_t n) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Rows of this CTA written as empty by one warp (capacity / range errors,
// empty key ranges): the O-CTAs write zero output, the S-CTAs lse = -inf.
__device__ void write_empty_warp(const Params& p, const Unit& u, uint32_t rank, int lane) {
  const int QH = p.Q * p.H;
  const long long total = (long long)p.B * QH;
  const int half = (int)(rank & 1u);
  if (rank >= 2) {
    for (int e = lane; e < kHM * 64; e += 32) {
      const int r = e >> 6, c = e & 63;
      const int lr = u.rt * kTM + half * kHM + r;
      if (lr >= QH) continue;
      const long long grow = (long long)u.b * QH + lr;
      __nv_bfloat16* dst = p.n_split == 1 ? p.out + grow * kC
                                          : p.part_o + ((long long)u.sp * total + grow) * kC;
      reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
    }
  } else {
    for (int r = lane; r < kHM; r += 32) {
      const int lr = u.rt * kTM + half * kHM + r;
      if (lr >= QH) continue;
      const long long grow = (long long)u.b * QH + lr;
      if (p.n_split == 1) {
        if (p.lse) p.lse[grow] = -INFINITY;
      } else {
        p.part_lse[(long long)u.sp * total + grow] = -INFINITY;
      }
    }
  }
}

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
__device__ void fused_write(const Params& p, int b, const unsigned char* bsm, int n, bool bad) {
  const TreeFuse& f = p.tf;
  const int32_t st = tb::write_warp(*reinterpret_cast<const tb::Smem*>(bsm), b, f.budget + 1, n,
                                    bad, f.tokens, f.parents, f.depths,
                                    reinterpret_cast<unsigned long long*>(f.vis_bits), f.vis,
                                    f.first_child, f.next_sibling, f.n_nodes);
  if ((threadIdx.x & 31) == 0 && st != 0) atomicOr(p.status + b, st);
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    k_verify_attn_pair(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ql,
                       const __grid_constant__ CUtensorMap tm_qp,
                       const __grid_constant__ CUtensorMap tm_o, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + N_BARS * 8);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };

  const uint32_t rank = cluster_rank();
  const bool s_side = rank < 2;
  const int half = (int)(rank & 1u);  // which 128 rows of the tile this CTA holds
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = (int)(gridDim.x >> 2);    // clusters of the launch
  const int cl = (int)(blockIdx.x >> 2);  // this cluster
  const long long U = (long long)p.B * p.n_rt * p.n_split;
  const int QH = p.Q * p.H;
  const long long total_rows = (long long)p.B * QH;
  const uint32_t vis_bytes = (uint32_t)(p.Q * kMaxW * 8);
  int32_t* order = reinterpret_cast<int32_t*>(smem + OFF_ORDER);
  UnitInfo* infos = reinterpret_cast<UnitInfo*>(smem + OFF_INFO);
  auto s_bt_of = [&](int i) { return reinterpret_cast<int32_t*>(smem + OFF_BT) + (i & 1) * kBtMax; };

  if (p.longest_first) {
    // Units are numbered by the rank of their sequence in (prefix length
    // descending, index ascending), found by every sequence counting the
    // sequences ahead of it; a long sequence then does not start last and
    // run alone at the end.
    int32_t* s_len = s_bt_of(0);  // the page buffers are free until the first unit
    if (tid < p.B) s_len[tid] = p.prefix_len[tid];
    __syncthreads();
    if (tid < p.B) {
      const int32_t mine = s_len[tid];
      int ahead = 0;
      for (int u = 0; u < p.B; ++u) {
        const int32_t o = s_len[u];
        ahead += (o > mine || (o == mine && u < tid)) ? 1 : 0;
      }
      order[ahead] = tid;
    }
    __syncthreads();
  }

  // ---- setup ---------------------------------------------------------------
  if (tid == 0) {
    if (s_side) {
      for (int s = 0; s < kStagesK * kKGroups; ++s) {
        mbar_init(bar(B_RING_FULL + s), 1);
        mbar_init(bar(B_RING_PEER + s), 1);
        mbar_init(bar(B_RING_EMPTY + s), 1);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(bar(B_S_FULL + s), 1);
        mbar_init(bar(B_S_EMPTY + s), 5);
        mbar_init(bar(B_S_READ + s), 4);
        mbar_init(bar(B_Q_FULL + s), 1);
        mbar_init(bar(B_Q_LOCAL + s), 1);
        mbar_init(bar(B_TREE + s), 1);
        mbar_init(bar(B_FIN_FREE + s), 4);
      }
      for (int s = 0; s < kMsgSlots; ++s) mbar_init(bar(B_P_FREE + s), 1);
      for (int s = 0; s < kStageSlots; ++s) mbar_init(bar(B_STAGE_FREE + s), 1);
      mbar_init(bar(B_Q_TMEM), 1);  // used on rank 0
      mbar_init(bar(B_Q_PEER), 1);  // used on rank 0
      mbar_init(bar(B_MMA_DONE), 2);
    } else {
      for (int s = 0; s < kStagesV; ++s) {
        mbar_init(bar(B_HALF_FULL + s), 1);
        mbar_init(bar(B_HALF_PEER + s), 1);
        mbar_init(bar(B_HALF_EMPTY + s), 1);
      }
      for (int s = 0; s < kMsgSlots; ++s) {
        mbar_init(bar(B_P_FULL + s), 1);
        mbar_init(bar(B_P_PEER + s), 1);
        mbar_init(bar(B_PV_DONE + s), 1);
      }
      mbar_init(bar(B_GO), 1);
      for (int s = 0; s < 2; ++s) {
        mbar_init(bar(B_O_READY + s), 4);
        mbar_init(bar(B_FIN_FULL + s), 1);
        mbar_init(bar(B_TAIL_OK + s), 2);
        mbar_init(bar(B_EPI_DONE + s), 8);
      }
      mbar_init(bar(B_OUT_FREE), 4);
      mbar_init(bar(B_MMA_DONE), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_INFO + s), 1);
      mbar_init(bar(B_INFO_FREE + s), s_side ? 10 : (rank == 2 ? 7 : 6));
    }
    fence_mbar_init();
    if (s_side) {
      // Q of the cluster's first unit depends on no check: it is loaded first.
      // q_lat comes in two halves, one per stage of the key ring, so that each
      // stage takes its first key tile as soon as its half is copied to TMEM;
      // q_pe goes to its own area, where it stays as an MMA operand.
      int b0, rt0, sp0;
      unit_coords(p, order, unit_id(cl, G, 0), &b0, &rt0, &sp0);
      const int row0 = (int)((long long)b0 * QH + (long long)rt0 * kTM + half * kHM);
      mbar_expect_tx(bar(B_Q_FULL + 0), kQlHalf + kQpBytes);
      tma_load_3d(sbase + S_RING, &tm_ql, 0, row0, 0, bar(B_Q_FULL + 0));
      tma_load_2d(sbase + S_QPE, &tm_qp, 0, row0, bar(B_Q_FULL + 0));
      mbar_expect_tx(bar(B_Q_FULL + 1), kQlHalf);
      tma_load_3d(sbase + S_RING + kTileK, &tm_ql, 0, row0, 4, bar(B_Q_FULL + 1));
    } else {
      for (int s = 0; s < kMsgSlots; ++s) {
        mbar_expect_tx(bar(B_P_FULL + s), kMsgBytes);
        if (rank == 2) mbar_expect_tx(bar(B_P_PEER + s), 16);  // rank 3's flags
      }
      for (int s = 0; s < 2; ++s) mbar_expect_tx(bar(B_FIN_FULL + s), kFinBytes);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  cluster_sync_after_init();  // every barrier and TMEM allocation of the cluster exists before any remote use

  bool failed = false;
  // the number of units of this cluster: one per full round, and one in the
  // last, partial round when its position there exists
  const int n_mine = (int)(U / G) + (unit_id(cl, G, (int)(U / G)) < U ? 1 : 0);
  // unit i of this cluster, as published by warp 0: 1 ready, 0 no such unit,
  // -1 the wait gave up
  auto take_unit = [&](int i, Unit& u) -> int {
    if (i >= n_mine) return 0;
    if (!mbar_wait(bar(B_INFO + (i & 1)), (i >> 1) & 1)) return -1;
    u = derive_unit(p, load_info(sbase + OFF_INFO + (i & 1) * sizeof(UnitInfo)));
    return 1;
  };
  // one thread per consuming warp
  auto release_unit = [&](int i) { mbar_arrive(bar(B_INFO_FREE + (i & 1))); };

  if (s_side) {
    // ========================= S-CTAs =========================
    if (warp == 0) {
      // ---- unit checks, then this CTA's Q and key halves (one TMA request each)
      if (lane == 0) prefetch_tmap(&tm_k);
      // Per-stage state in bit fields (bit s: stage s), kept in registers:
      // rpar the parity of the key halves loaded into the stage, keyl whether
      // its last user is a key half (else a Q half), qused whether that Q half
      // was copied to TMEM (by a unit of parity bit s of lqpar; else it was never
      // used); tpar / tused the building units per ancestor-word buffer.
      int kq = 0;  // units with key tiles so far
      int qn = 1;  // Q loads issued (the first unit's at setup)
      uint32_t rpar = 0, keyl = 0, qused = 0, lqpar = 0, tpar = 0, tused = 0;
      for (int i = 0; !failed; ++i) {
        const long long uid = unit_id(cl, G, i);
        if (uid >= U) break;
        if (i >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(bar(B_INFO_FREE + (i & 1)), ((i >> 1) - 1) & 1))) {
          failed = true;
          break;
        }
        int b, rt, sp;
        unit_coords(p, order, uid, &b, &rt, &sp);
        unit_checks(p, b, rt, sp, s_bt_of(i), infos + (i & 1), lane);
        if (lane == 0) mbar_arrive(bar(B_INFO + (i & 1)));
        const Unit u = derive_unit(p, load_info(sbase + OFF_INFO + (i & 1) * sizeof(UnitInfo)));
        if (u.nt == 0) {
          write_empty_warp(p, u, rank, lane);
          if (u.code && u.rt == 0 && u.sp == 0 && rank == 0 && lane == 0)
            atomicOr(p.status + u.b, u.code);
          continue;
        }
        int ok = 1;
        if (lane == 0) {
          if (u.builds) {
            mbar_expect_tx(bar(B_TREE + (kq & 1)), vis_bytes);
            tpar ^= 1u << (kq & 1);
            tused |= 1u << (kq & 1);
          }
          if (i > 0) {
            // the unit's Q goes into both stages once their last user is done:
            // the MMAs of a key half (which also ends the previous unit's reads
            // of q_pe and of the q_lat in TMEM), a Q half copied to TMEM, or a
            // Q load that was never used
            for (int s = 0; s < 2 && ok; ++s)
              ok = (keyl >> s) & 1 ? mbar_wait_cluster(bar(B_RING_EMPTY + s * kKGroups + kKGroups - 1),
                                                       ((rpar >> s) & 1) ^ 1)
                   : (qused >> s) & 1 ? mbar_wait(bar(B_Q_LOCAL + s), (lqpar >> s) & 1)
                                      : mbar_wait(bar(B_Q_FULL + s), (qn - 1) & 1);
            if (ok) {
              const int row0 = (int)((long long)u.b * QH + (long long)u.rt * kTM + half * kHM);
              mbar_expect_tx(bar(B_Q_FULL + 0), kQlHalf + kQpBytes);
              tma_load_3d(sbase + S_RING, &tm_ql, 0, row0, 0, bar(B_Q_FULL + 0));
              tma_load_2d(sbase + S_QPE, &tm_qp, 0, row0, bar(B_Q_FULL + 0));
              mbar_expect_tx(bar(B_Q_FULL + 1), kQlHalf);
              tma_load_3d(sbase + S_RING + kTileK, &tm_ql, 0, row0, 4, bar(B_Q_FULL + 1));
              ++qn;
            }
          }
          keyl = 0;
          qused = 3;
          lqpar = (kq & 1) ? 3u : 0u;
          const int32_t* s_bt = s_bt_of(i);
          for (int uu = 0; uu < u.nt && ok; ++uu) {
            const int slot = uu & 1;
            // The stage is free once its half of q_lat has left it; later a
            // chunk of the stage is reloaded as soon as the MMAs of the tile
            // two back have read it, so the next tile's keys are in place
            // long before its MMAs start.
            if (uu < 2 && !mbar_wait(bar(B_Q_LOCAL + slot), kq & 1)) {
              ok = 0;
              break;
            }
            int blk = 2 * tile_of(u, uu) + half;
            if (blk >= u.n_blocks) blk -= 1;  // the phantom half: the other half's rows
            const int krow = (int)block_row(p, u, s_bt, blk);
            const int gb0 = slot * kKGroups;
            for (int q = 0; q < kKGroups; ++q) {
              if (uu >= 2 &&
                  !mbar_wait_cluster(bar(B_RING_EMPTY + gb0 + q), ((rpar >> slot) & 1) ^ 1)) {
                ok = 0;
                break;
              }
              mbar_expect_tx(bar(B_RING_FULL + gb0 + q), kGroupChunks * kKChunk);
              tma_load_3d(sbase + S_RING + slot * kTileK + q * kGroupChunks * kKChunk, &tm_k, 0,
                          krow, q * kGroupChunks, bar(B_RING_FULL + gb0 + q));
            }
            rpar ^= 1u << slot;
            keyl |= 1u << slot;
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) failed = true;
        ++kq;
      }
      // nothing may land after the CTAs leave
      if (lane == 0) {
        for (int s = 0; s < 2; ++s) {
          bool ok = true;
          if ((keyl >> s) & 1) {
            for (int q = 0; q < kKGroups; ++q)
              ok = mbar_wait(bar(B_RING_FULL + s * kKGroups + q), ((rpar >> s) & 1) ^ 1) && ok;
          } else {
            ok = mbar_wait(bar(B_Q_FULL + s), (qn - 1) & 1);
          }
          if (!ok) failed = true;
          if (((tused >> s) & 1) && !mbar_wait_cluster(bar(B_TREE + s), ((tpar >> s) & 1) ^ 1))
            failed = true;
        }
      }
    } else if (rank == 0 && (warp == 1 || warp == 10)) {
      // QK^T for both S-CTAs over 128 keys: q_lat from TMEM (TS), q_pe from
      // shared memory (SS), B = the two 64-key halves, D = S (128 x 128 in
      // each CTA). Tile jj of a unit uses S buffer and key stage jj & 1, and
      // issuer jj & 1 (warp 1: even tiles, warp 10: odd tiles).
      if (lane == 0) {
        const int sb = warp == 1 ? 0 : 1;
        int kq = 0, n_iss = 0;  // tiles this issuer has issued (uses of its stage and S buffer)
        int qn = 0;             // Q loads consumed (the first unit's counts even without tiles)
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          if (t < 0) {
            failed = true;
            break;
          }
          if (u.nt == 0 && i == 0) qn = 1;
          if (u.nt > 0) {
            bool ok;
            if (sb == 0) {
              // The unit's q_lat, staged in both stages of the key ring of both
              // CTAs, goes to TMEM columns [0, 256) (bf16 pairs, row = lane)
              // through the tensor pipe, ahead of the first MMAs, which see it
              // in issue order; each stage is handed back to its producer once
              // its copies are done. The previous unit's MMAs, the last readers
              // of those columns, completed before the producers loaded this Q.
              ok = mbar_wait(bar(B_Q_FULL + 0), qn & 1) && mbar_wait(bar(B_Q_FULL + 1), qn & 1) &&
                   mbar_wait_cluster(bar(B_Q_PEER), kq & 1);
              tc_fence_after();
              if (ok) {
#pragma unroll 1
                for (int s = 0; s < 2; ++s) {
                  const uint32_t qs = sbase + S_RING + s * kTileK;
#pragma unroll
                  for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                      tmem_cp_pair_128x256b(
                          tmem + kTmemQ + 32 * (4 * s + c) + 8 * kk,
                          smem_desc(qs + c * (kHM * 128) + kk * 32, 16, 1024, kSwizzle128B));
                  umma_pair_commit(bar(B_Q_LOCAL + s), kMaskS);
                }
                umma_pair_commit(bar(B_Q_TMEM), 0x1);
              }
            } else {
              ok = mbar_wait_cluster(bar(B_Q_TMEM), kq & 1);
              tc_fence_after();
            }
            ++qn;
            for (int jj = sb; jj < u.nt && ok; jj += 2) {
              if (n_iss > 0 && !mbar_wait_cluster(bar(B_S_EMPTY + sb), (n_iss - 1) & 1)) {
                ok = false;
                break;
              }
              const uint32_t d = tmem + kTmemS + sb * kBS;
              const uint32_t st = sbase + S_RING + sb * kTileK;
              const int gb0 = sb * kKGroups;
              // group by group: each is waited for (here and on rank 1) and
              // released to the producer as soon as its MMAs are done
#pragma unroll 1
              for (int q = 0; q < kKGroups && ok; ++q) {
                if (!mbar_wait(bar(B_RING_FULL + gb0 + q), n_iss & 1) ||
                    !mbar_wait_cluster(bar(B_RING_PEER + gb0 + q), n_iss & 1)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < kGroupChunks; ++cc) {
                  const int c = q * kGroupChunks + cc;
                  if (c < kC / 64) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                      const uint64_t bd =
                          smem_desc(st + c * kKChunk + kk * 32, 16, 1024, kSwizzle128B);
                      umma_pair_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * kk, bd, kIdescS,
                                        (c | kk) ? 1u : 0u);
                    }
                  } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                      const uint64_t ad =
                          smem_desc(sbase + S_QPE + kk * 32, 16, 1024, kSwizzle128B);
                      const uint64_t bd =
                          smem_desc(st + c * kKChunk + kk * 32, 16, 1024, kSwizzle128B);
                      umma_pair_bf16(d, ad, bd, kIdescS, 1u);
                    }
                  }
                }
                umma_pair_commit(bar(B_RING_EMPTY + gb0 + q), kMaskS);
              }
              if (!ok) break;
              umma_pair_commit(bar(B_S_FULL + sb), kMaskS);
              ++n_iss;
            }
            if (!ok) {
              failed = true;
              break;
            }
            ++kq;
          }
          release_unit(i);
        }
        umma_pair_commit(bar(B_MMA_DONE), 0x1);
        if (!mbar_wait(bar(B_MMA_DONE), 0)) failed = true;
      }
    } else if (rank == 1 && warp == 10) {
      // relay: this CTA's Q, then each key half of a tile, has landed -> rank
      // 0's MMA issuers (each CTA's tile loads complete on its own barrier; a
      // load that signals the peer's barrier directly slows this CTA's
      // outgoing P copies)
      if (lane == 0) {
        const uint32_t peer0 = map_peer(bar(B_RING_PEER), 0);
        uint32_t par = 0;  // bit s: parity of the key halves of stage s
        int qn = 0;        // Q loads consumed (the first unit's counts even without tiles)
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          bool ok = t > 0;
          if (ok && u.nt == 0 && i == 0) qn = 1;
          if (ok && u.nt > 0) {
            ok = mbar_wait(bar(B_Q_FULL + 0), qn & 1) && mbar_wait(bar(B_Q_FULL + 1), qn & 1);
            if (ok) mbar_arrive_cluster_relaxed(map_peer(bar(B_Q_PEER), 0));
            ++qn;
          }
          for (int uu = 0; ok && uu < u.nt; ++uu) {
            const int slot = uu & 1;
            for (int q = 0; ok && q < kKGroups; ++q) {
              ok = mbar_wait(bar(B_RING_FULL + slot * kKGroups + q), (par >> slot) & 1);
              if (ok) mbar_arrive_cluster_relaxed(peer0 + 8 * (slot * kKGroups + q));
            }
            par ^= 1u << slot;
          }
          if (!ok) {
            failed = true;
            break;
          }
          release_unit(i);
        }
      }
    } else if (rank == 1 && warp == 1) {
      // relay: this CTA's group has read an S buffer -> rank 0's MMA issuers
      // (the softmax warps arrive locally; a release at cluster scope from each
      // of them held them up for about a microsecond per tile)
      if (lane == 0) {
        const uint32_t s_empty0 = map_peer(bar(B_S_EMPTY), 0);
        uint32_t par = 0;  // bit s: parity of the reads of S buffer s
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          bool ok = t > 0;
          for (int jj = 0; ok && jj < u.nt; ++jj) {
            const int sb = jj & 1;
            ok = mbar_wait(bar(B_S_READ + sb), (par >> sb) & 1);
            par ^= 1u << sb;
            if (ok) mbar_arrive_cluster_relaxed(s_empty0 + 8 * sb);
          }
          if (!ok) {
            failed = true;
            break;
          }
          release_unit(i);
        }
      }
    } else if (warp >= 2 && warp <= 9) {
      // ---------------- softmax: two groups of four warps, alternate tiles ----
      // Group g (warps 2-5: g = 0, warps 6-9: g = 1) takes the tiles jj of a
      // unit with jj % 2 == g (so also S buffer g), one thread per row over
      // all 128 keys. The only thing that passes from tile to tile is each
      // row's running max, handed from one group to the other through shared
      // memory and a named barrier per (lane quadrant, direction); the
      // exponentials of consecutive tiles run in the two groups at once.
      // Every handoff is made whatever happens (a group that gave up on a
      // wait skips its work, not its barriers), so neither group can be left
      // waiting for the other; the eight warps leave the unit loop together.
      const int qd = warp & 3;
      const int g = (warp - 2) >> 2;
      const int r = qd * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
      const int W = (p.Q + 63) >> 6;
      const uint32_t hand = sbase + S_XCH;     // float [row]: running max handoff
      const uint32_t fin = hand + kHM * 4;     // float [group][row][2]: (m, l) at the end
      const uint32_t msg_peer0 = map_peer(sbase + O_MSG, rank + 2);
      const uint32_t pfull_peer0 = map_peer(bar(B_P_FULL), rank + 2);
      const uint32_t bar_in = 2 + 2 * qd + g;         // handoff to this group
      const uint32_t bar_out = 2 + 2 * qd + (g ^ 1);  // handoff to the other group
      const uint32_t bar_grp = 10 + g;                // the group's four warps
      const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
      // Counters carried from unit to unit, kept in shared memory (the tile
      // loop needs every register): [0] units with key tiles so far, [1] bit
      // v the parity of the building units of ancestor-word buffer v, [2]
      // tiles this group took in the earlier units (uses of S buffer g), [3]
      // P blocks of the earlier units.
      const uint32_t cnt = sbase + OFF_CNT + 32 * (warp - 2);  // int32 [8]
      auto cnt_ld = [&](int k) { return lds_s32(cnt + 4 * k); };
      auto cnt_st = [&](int k, int v) { sts_s32(cnt + 4 * k, v); };
      if (lane == 0)
        for (int k = 0; k < 4; ++k) cnt_st(k, 0);
      __syncwarp();
      for (int i = 0; !failed; ++i) {
        Unit u;
        const int t = take_unit(i, u);
        if (t == 0) break;  // the same for all eight warps
        if (!bar1_and(t > 0, 256)) {
          failed = true;
          break;
        }
        if (u.nt == 0) {
          __syncwarp();
          if (lane == 0) release_unit(i);
          continue;
        }
        const int lr = u.rt * kTM + half * kHM + r;
        const bool row_ok = lr < QH;
        const int qi = row_ok ? lr / p.H : 0;
        // The row's ancestor words sit in the unit's buffer of S_VIS (filled by
        // the fused build, or here from the caller's vis_bits: each thread
        // writes the words of its own query, which it alone reads back), and
        // are read where a block holds tree keys.
        const uint32_t vis_row =
            sbase + S_VIS + (cnt_ld(0) & 1) * kVisBuf +
            (DDT_GUARD(qi < p.Q, 103, p.status + u.b) ? qi : 0) * kMaxW * 8;
        if (!p.fuse && row_ok) {
          const unsigned long long* vb = p.vis_bits + ((size_t)u.b * p.Q + qi) * W;
          sts_u64(vis_row, vb[0]);
          sts_u64(vis_row + 8, W > 1 ? vb[1] : 0ull);
        }
        const int Lk = (int)u.L;       // prefix keys
        const int nk_all = (int)u.n_keys;

        float m_run = -INFINITY;  // the row's running max (scaled, log2 units)
        float m_l = -INFINITY;    // reference max of this group's partial sum
        float l_run = 0.f;        // this group's share of the row sum, relative to m_l
        int rj = u.rot;
        for (int jj = 0; jj < u.nt; ++jj) {
          const int tile = jj < u.nrot ? u.j_begin + rj : u.j_begin + jj;
          if (jj < u.nrot && ++rj == u.nrot) rj = 0;
          if ((jj & 1) != g) continue;
          bool ok = !failed;
          float x[128];  // raw scores q.k of the tile's 128 keys
          if (ok) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait_cluster(bar(B_S_FULL + g), (cnt_ld(2) + (jj >> 1)) & 1));
            tc_fence_after();
            uint32_t sa[128];  // the whole S row in one request, so the buffer is freed soon
            tmem_ld128(t_lane + kTmemS + g * kBS, sa);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 128; ++k) x[k] = __uint_as_float(sa[k]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar((rank == 0 ? B_S_EMPTY : B_S_READ) + g));
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              const int blk = 2 * tile + kb;
              const int t0 = blk * kBK;
              unsigned long long m = ~0ull;  // visible keys of the block
              if (blk >= u.n_blocks) {
                m = 0ull;  // the phantom block
              } else if (t0 + kBK > Lk) {
                if (p.fuse) {
                  const int vb = cnt_ld(0) & 1;
                  ok = ok && __all_sync(0xffffffffu, mbar_wait_cluster(bar(B_TREE + vb),
                                                                        (cnt_ld(1) >> vb) & 1));
                }
                const unsigned long long vis0 = row_ok ? lds_u64(vis_row) : 0ull;
                const unsigned long long vis1 = row_ok ? lds_u64(vis_row + 8) : 0ull;
                // key k is slot t0 + k; slots below L are prefix, slot L + t is
                // tree slot t (bit t of vis1:vis0), slots from n_keys on do not exist
                const int np = max(0, Lk - t0);
                const int off = t0 - Lk;
                const int nk = min(64, nk_all - t0);
                unsigned long long tm;
                if (off < 0) tm = vis0 << (-off);
                else if (off == 0) tm = vis0;
                else if (off < 64) tm = (vis0 >> off) | (vis1 << (64 - off));
                else tm = vis1 >> (off - 64);
                const unsigned long long pm = (1ull << np) - 1ull;
                const unsigned long long km = nk >= 64 ? ~0ull : (1ull << nk) - 1ull;
                m = (pm | tm) & km;
              }
              if (m != ~0ull) {
#pragma unroll
                for (int k = 0; k < 64; ++k)
                  if (!((m >> k) & 1ull)) x[64 * kb + k] = -INFINITY;
              }
            }
          }
          float mt = -INFINITY;
          if (ok) {
            float mx8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mx8[q] = x[q];
#pragma unroll
            for (int k = 8; k < 128; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], x[k]);
            // the scale is positive, so it commutes with the max
            mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                 p.scale_log2;
          }
          // running max after the previous tile, from the other group
          if (jj > 0) {
            asm volatile("bar.sync %0, 64;" ::"r"(bar_in) : "memory");
            m_run = lds_f32(hand + 4 * r);
          }
          // lazy rescale: the reference max moves only when the row max passes it
          // by 8 (a factor 2^8); O on the peer is then multiplied by `factor`
          // before the tile's first block is added
          float factor = 1.f;
          bool rescale = false;
          if (mt > m_run + 8.f) {
            factor = ex2(m_run - mt);  // 0 when m_run is -inf
            rescale = jj > 0;
            m_run = mt;
          }
          if (jj + 1 < u.nt) {
            sts_f32(hand + 4 * r, m_run);
            asm volatile("bar.arrive %0, 64;" ::"r"(bar_out) : "memory");
          }
          // Exponentials, P blocks and their copies. The group barriers run
          // whatever `ok` is (a warp that gave up skips the work, not the
          // barriers); the phantom block is skipped by the whole group.
          if (ok && m_run != m_l) {
            if (l_run != 0.f) l_run *= ex2(m_l - m_run);
            m_l = m_run;
          }
          // p = 2^(x * scale*log2(e) - m); every x is -inf while m is -inf: p = 0
          const float nm = m_run == -INFINITY ? 0.f : -m_run;
          const float2 neg_m = make_float2(nm, nm);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            if (2 * tile + kb >= u.n_blocks) continue;
            const int msg_g = cnt_ld(3) + 2 * jj + kb;  // the P block's number in the cluster's stream
            const int ss = msg_g % kStageSlots;
            if (ok && msg_g >= kStageSlots)
              ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(B_STAGE_FREE + ss),
                                                             ((msg_g / kStageSlots) - 1) & 1));
            if (ok) {
              unsigned char* msg = smem + S_STAGE + ss * kMsgStride;
              const uint32_t p_row =
                  sbase + S_STAGE + ss * kMsgStride + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
              for (int c = 0; c < 8; ++c) {  // 8 keys -> one 16-byte unit of the row
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int k = 64 * kb + 8 * c + 2 * e;
                  const float2 ex = ffma2(make_float2(x[k], x[k + 1]), sl2, neg_m);
                  const float2 pp = make_float2(ex2(ex.x), ex2(ex.y));
                  pk[e] = pack_bf16(pp.x, pp.y);
                  acc[e] = fadd2(acc[e], pp);
                }
                const uint32_t addr = p_row + ((uint32_t)(c ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[0]),
                             "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                             : "memory");
              }
              // the rescale travels with the tile's first block only
              if (kb == 0) reinterpret_cast<float*>(msg + kPBytes)[r] = rescale ? factor : 1.f;
              const bool any_rescale = kb == 0 && __any_sync(0xffffffffu, rescale);
              if (lane == 0) reinterpret_cast<uint32_t*>(msg + kPBytes + kHM * 4)[qd] = any_rescale;
              fence_proxy_async_smem();
            }
            // the group's four warps have written the block: one thread sends it,
            // once PV has released the O-CTA slot it goes to
            const bool all_ok = bar1_and_id(ok, bar_grp, 128);
            if (!all_ok) ok = false;
            if (all_ok && lane == 0 && warp == 2 + 4 * g) {
              const int mb = msg_g % kMsgSlots;
              if (msg_g < kMsgSlots ||
                  mbar_wait_cluster(bar(B_P_FREE + mb), ((msg_g / kMsgSlots) - 1) & 1))
                bulk_copy_to_peer(msg_peer0 + mb * kMsgStride, sbase + S_STAGE + ss * kMsgStride,
                                  kMsgBytes, pfull_peer0 + 8 * mb);
              else
                ok = false;
            }
          }
          if (ok) {
            const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
            l_run += a.x + a.y;
          }
          // a wait that gave up in any warp of the group stops the whole group
          if (!bar1_and_id(ok, bar_grp, 128)) failed = true;
        }

        // ---- the unit's end: the row sum over both groups, lse here, 1/l to
        // the O-CTA (through one of two buffers, by unit parity) ------------
        const Unit ue = derive_unit(p, load_info(sbase + OFF_INFO + (i & 1) * sizeof(UnitInfo)));
        sts_f32x2(fin + 8 * (g * kHM + r), m_l, l_run);
        asm volatile("bar.sync %0, 64;" ::"r"(12 + qd) : "memory");
        bool fin_ok = bar1_and(!failed, 256);
        const int kq = cnt_ld(0);
        const int fb = kq & 1;
        if (g == 0 && fin_ok && kq >= 2)  // the O-CTA has read this buffer's previous 1/l
          fin_ok = __all_sync(0xffffffffu,
                              mbar_wait_cluster(bar(B_FIN_FREE + fb), ((kq >> 1) - 1) & 1));
        if (g == 0 && fin_ok) {
          const float2 fa = lds_f32x2(fin + 8 * r), fb2 = lds_f32x2(fin + 8 * (kHM + r));
          const float ma = fa.x, la = fa.y, mb2 = fb2.x, lb = fb2.y;
          const float mf = fmaxf(ma, mb2);
          float l_tot = 0.f;
          if (la != 0.f) l_tot += la * ex2(ma - mf);
          if (lb != 0.f) l_tot += lb * ex2(mb2 - mf);
          const bool live = l_tot > 0.f;
          const int lre = ue.rt * kTM + half * kHM + r;
          const long long grow = (long long)ue.b * QH + lre;
          if (lre < QH) {
            const float lse_v = live ? (mf + __log2f(l_tot)) * 0.69314718055994530942f : -INFINITY;
            if (!DDT_GUARD(grow < total_rows, 104, p.status + ue.b)) {
            } else if (p.n_split == 1) {
              if (p.lse) p.lse[grow] = lse_v;
            } else {
              p.part_lse[(long long)ue.sp * total_rows + grow] = lse_v;
            }
          }
          reinterpret_cast<float*>(smem + S_FIN + fb * kFinBytes)[r] = live ? 1.f / l_tot : 0.f;
          fence_proxy_async_smem();
        }
        fin_ok = bar1_and(fin_ok, 256);
        if (tid == 64 && fin_ok)
          bulk_copy_to_peer(map_peer(sbase + O_FIN + fb * kFinBytes, rank + 2),
                            sbase + S_FIN + fb * kFinBytes, kFinBytes,
                            map_peer(bar(B_FIN_FULL + fb), rank + 2));
        if (!fin_ok) {
          failed = true;
        }
        if (lane == 0) release_unit(i);
        __syncwarp();
        if (lane == 0) {
          if (ue.builds) cnt_st(1, cnt_ld(1) ^ (1 << (kq & 1)));
          cnt_st(0, kq + 1);
          cnt_st(2, cnt_ld(2) + (ue.nt - g + 1) / 2);
          cnt_st(3, cnt_ld(3) + ue.n_msgs);
        }
        __syncwarp();
      }
    }
  } else {
    // ========================= O-CTAs =========================
    if (warp == 0) {
      // ---- unit checks, then this CTA's 256 value dims of each block (one
      // request each), and the zeroed tail of the unit's last block
      if (lane == 0) prefetch_tmap(&tm_v);
      int kq = 0;
      uint32_t vpar = 0, vused = 0;  // bit s: parity of the value halves of stage s, stage used
      for (int i = 0; !failed; ++i) {
        const long long uid = unit_id(cl, G, i);
        if (uid >= U) break;
        if (i >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(bar(B_INFO_FREE + (i & 1)), ((i >> 1) - 1) & 1))) {
          failed = true;
          break;
        }
        int b, rt, sp;
        unit_coords(p, order, uid, &b, &rt, &sp);
        unit_checks(p, b, rt, sp, s_bt_of(i), infos + (i & 1), lane);
        if (lane == 0) mbar_arrive(bar(B_INFO + (i & 1)));
        const Unit u = derive_unit(p, load_info(sbase + OFF_INFO + (i & 1) * sizeof(UnitInfo)));
        if (u.nt == 0) {
          write_empty_warp(p, u, rank, lane);
          continue;
        }
        int ok = 1;
        if (lane == 0) {
          const int32_t* s_bt = s_bt_of(i);
          for (int m = 0; m < u.n_msgs; ++m) {
            const int stage = m % kStagesV;
            if (((vused >> stage) & 1) &&
                !mbar_wait_cluster(bar(B_HALF_EMPTY + stage), ((vpar >> stage) & 1) ^ 1)) {
              ok = 0;
              break;
            }
            // the previous unit's output is staged in stage 2
            if (m == 2 && kq > 0 && !mbar_wait(bar(B_OUT_FREE), (kq - 1) & 1)) {
              ok = 0;
              break;
            }
            mbar_expect_tx(bar(B_HALF_FULL + stage), kTileV);
            tma_load_4d(sbase + O_RING + stage * kTileV, &tm_v, 0,
                        (int)block_row(p, u, s_bt, msg_block(u, m)), 2 * half, 0,
                        bar(B_HALF_FULL + stage));
            vpar ^= 1u << stage;
            vused |= 1u << stage;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
          // keys past the end of the sequence in the last block: their values are
          // zeroed so that 0 * (whatever the page holds) cannot turn into NaN
          const int m = u.n_msgs - 1;
          const int stage = m % kStagesV;
          const long long t0 = (long long)msg_block(u, m) * kBK;
          if (t0 + kBK > u.n_keys) {
            // the stage parities live in lane 0, which issued the loads
            const uint32_t ph = __shfl_sync(0xffffffffu, ((vpar >> stage) & 1) ^ 1, 0);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_HALF_FULL + stage), ph));
            if (ok) {
              unsigned char* base = smem + O_RING + stage * kTileV;
              const int r0 = (int)(u.n_keys - t0);
              for (int e = lane; e < (kBK - r0) * 32; e += 32) {  // 16-byte units, 4 chunks
                const int rr = r0 + (e >> 5), c = (e >> 3) & 3, q = e & 7;
                reinterpret_cast<uint4*>(base + c * kVChunk + (rr >> 3) * 1024 + (rr & 7) * 128)[q] =
                    make_uint4(0, 0, 0, 0);
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (ok && lane == 0) {
            if (rank == 2) mbar_arrive(bar(B_TAIL_OK + (kq & 1)));
            else mbar_arrive_cluster(map_peer(bar(B_TAIL_OK + (kq & 1)), 2));
          }
        }
        if (!ok) {
          failed = true;
        }
        ++kq;
      }
      // nothing may land after the CTAs leave
      if (lane == 0)
        for (int s = 0; s < kStagesV; ++s)
          if (((vused >> s) & 1) && !mbar_wait(bar(B_HALF_FULL + s), ((vpar >> s) & 1) ^ 1))
            failed = true;
    } else if (warp == 1 && rank == 2) {
      if (lane == 0) {  // PV for both O-CTAs: A = P (K-major), B = value halves (MN-major)
        // Before PV of message jj the O rows of a quadrant whose flag is set in
        // the message are multiplied by the row's factor; this thread reads the
        // flags of both CTAs' messages and calls the row warps only then. The
        // first PV of a unit overwrites O, once both CTAs' row warps have read
        // the previous unit's O.
        const uint32_t go3 = map_peer(bar(B_GO), 3);
        const uint32_t goidx3 = map_peer(sbase + O_GO, 3);
        uint32_t n_go2 = 0, n_go3 = 0;  // completed rescale calls per CTA
        int kq = 0, gb = 0;
        uint32_t vpar = 0;  // bit s: parity of the value halves of stage s
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          if (t < 0) {
            failed = true;
            break;
          }
          if (u.nt > 0) {
            bool ok = true;
            for (int jj = 0; jj < u.n_msgs && ok; ++jj) {
              const int mg = gb + jj;
              const int mb = mg % kMsgSlots;
              const uint32_t ph = (mg / kMsgSlots) & 1;
              const int stage = jj % kStagesV;
              const uint32_t vph = (vpar >> stage) & 1;
              vpar ^= 1u << stage;
              if (!mbar_wait(bar(B_P_FULL + mb), ph) || !mbar_wait_cluster(bar(B_P_PEER + mb), ph)) {
                ok = false;
                break;
              }
              // rank 3's flags of the slot's next message complete the next phase
              mbar_expect_tx(bar(B_P_PEER + mb), 16);
              if (jj > 0) {
                const uint4 f2 = *reinterpret_cast<const uint4*>(smem + O_MSG + mb * kMsgStride +
                                                                 kPBytes + kHM * 4);
                const uint4 f3 = *reinterpret_cast<const uint4*>(smem + O_PEERFLAG + 16 * mb);
                const bool r2 = (f2.x | f2.y | f2.z | f2.w) != 0;
                const bool r3 = (f3.x | f3.y | f3.z | f3.w) != 0;
                if (r2 || r3) {
                  // O is rescaled once PV of the previous message has completed
                  const int pm = mg - 1;
                  if (!mbar_wait(bar(B_PV_DONE + pm % kMsgSlots), (pm / kMsgSlots) & 1)) {
                    ok = false;
                    break;
                  }
                  if (r2) {
                    *reinterpret_cast<volatile int32_t*>(smem + O_GO) = jj;
                    mbar_arrive(bar(B_GO));
                  }
                  if (r3) {
                    st_cluster_u32(goidx3, (uint32_t)jj);
                    mbar_arrive_cluster(go3);
                  }
                  if ((r2 && !mbar_wait(bar(B_O_READY + 0), n_go2++ & 1)) ||
                      (r3 && !mbar_wait_cluster(bar(B_O_READY + 1), n_go3++ & 1))) {
                    ok = false;
                    break;
                  }
                }
              } else if (kq > 0 &&
                         !mbar_wait_cluster(bar(B_EPI_DONE + ((kq - 1) & 1)), ((kq - 1) >> 1) & 1)) {
                ok = false;
                break;
              }
              if (!mbar_wait(bar(B_HALF_FULL + stage), vph) ||
                  !mbar_wait_cluster(bar(B_HALF_PEER + stage), vph) ||
                  (jj == u.n_msgs - 1 &&
                   !mbar_wait_cluster(bar(B_TAIL_OK + (kq & 1)), (kq >> 1) & 1))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t pa = sbase + O_MSG + mb * kMsgStride;
              const uint32_t h0 = sbase + O_RING + stage * kTileV;
              const uint32_t h1 = h0 + 2 * kVChunk;
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint64_t ad = smem_desc(pa + kk * 32, 16, 1024, kSwizzle128B);
                const uint32_t acc = (jj > 0 || kk > 0) ? 1u : 0u;
                umma_pair_bf16(tmem, ad, smem_desc(h0 + kk * 2048, kVChunk, 1024, kSwizzle128B),
                               kIdescPV, acc);
                umma_pair_bf16(tmem + 256, ad,
                               smem_desc(h1 + kk * 2048, kVChunk, 1024, kSwizzle128B), kIdescPV,
                               acc);
              }
              umma_pair_commit(bar(B_PV_DONE + mb), kMaskO);
              umma_pair_commit(bar(B_HALF_EMPTY + stage), kMaskO);
              umma_pair_commit(bar(B_P_FREE + mb), kMaskS);
            }
            // the row warps of both CTAs leave their call loop (even after a failure)
            *reinterpret_cast<volatile int32_t*>(smem + O_GO) = -1;
            mbar_arrive(bar(B_GO));
            st_cluster_u32(goidx3, 0xffffffffu);
            mbar_arrive_cluster(go3);
            if (!ok) {
              failed = true;
              break;
            }
            gb += u.n_msgs;
            ++kq;
          }
          release_unit(i);
        }
        umma_pair_commit(bar(B_MMA_DONE), 0x4);
        if (!mbar_wait(bar(B_MMA_DONE), 0)) failed = true;
      }
    } else if (rank == 3 && warp == 8) {
      // relay: this CTA's value half of a block has landed -> rank 2's PV issuer
      if (lane == 0) {
        const uint32_t peer2 = map_peer(bar(B_HALF_PEER), 2);
        uint32_t par = 0;  // bit s: parity of the value halves of stage s
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          bool ok = t > 0;
          for (int m = 0; ok && u.nt > 0 && m < u.n_msgs; ++m) {
            const int stage = m % kStagesV;
            ok = mbar_wait(bar(B_HALF_FULL + stage), (par >> stage) & 1);
            par ^= 1u << stage;
            if (ok) mbar_arrive_cluster_relaxed(peer2 + 8 * stage);
          }
          if (!ok) {
            failed = true;
            break;
          }
          release_unit(i);
        }
      }
    } else if (warp == 7) {
      // ---------------- relay: incoming messages --------------------------------
      // Once a message has landed here: arm its slot for the slot's next
      // message, free the S-CTA's staging slot it came from, and (rank 3)
      // tell rank 2's PV issuer.
      if (lane == 0) {
        const uint32_t stage_free0 = map_peer(bar(B_STAGE_FREE), rank - 2);
        const uint32_t ppeer2 = map_peer(bar(B_P_PEER), 2);
        int gb = 0;
        for (int i = 0; !failed; ++i) {
          Unit u;
          const int t = take_unit(i, u);
          if (t == 0) break;
          bool ok = t > 0;
          for (int jj = 0; ok && u.nt > 0 && jj < u.n_msgs; ++jj) {
            const int mg = gb + jj;
            const int mb = mg % kMsgSlots;
            ok = mbar_wait_cluster(bar(B_P_FULL + mb), (mg / kMsgSlots) & 1);
            if (!ok) break;
            mbar_expect_tx(bar(B_P_FULL + mb), kMsgBytes);
            mbar_arrive_cluster_relaxed(stage_free0 + 8 * (mg % kStageSlots));
            if (rank == 3) {
              // the relay to rank 2's PV issuer carries the message's rescale
              // flags: one 16-byte asynchronous store that completes rank 2's
              // P_PEER phase on arrival (so the issuer reads them locally)
              const uint4 fl = *reinterpret_cast<const uint4*>(smem + O_MSG + mb * kMsgStride +
                                                               kPBytes + kHM * 4);
              st_async_v4(map_peer(sbase + O_PEERFLAG, 2) + 16 * mb, fl.x, fl.y, fl.z, fl.w,
                          ppeer2 + 8 * mb);
            }
          }
          if (!ok) {
            failed = true;
            break;
          }
          if (u.nt > 0) gb += u.n_msgs;
          release_unit(i);
        }
      }
    } else if (warp >= 2 && warp <= 5) {
      // ---------------- row warps: rescales when called, output ---------------
      const int qd = warp & 3;
      const int r = qd * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
      const uint32_t oready = rank == 2 ? bar(B_O_READY + 0) : map_peer(bar(B_O_READY + 1), 2);
      const uint32_t epi_done = rank == 2 ? bar(B_EPI_DONE) : map_peer(bar(B_EPI_DONE), 2);
      const uint32_t fin_free = map_peer(bar(B_FIN_FREE), rank - 2);
      const uint32_t box_w = sbase + O_OUT + (uint32_t)qd * 2 * kOutBox;  // this warp's two boxes
      int kq = 0, gb = 0;
      uint32_t gcall = 0;  // GO calls so far
      for (int i = 0; !failed; ++i) {
        Unit u;
        const int t = take_unit(i, u);
        if (t == 0) break;
        if (t < 0) {
          failed = true;
          break;
        }
        if (u.nt > 0) {
          const int lr = u.rt * kTM + half * kHM + r;
          const bool row_ok = lr < QH;
          const long long row0 = (long long)u.b * QH + (long long)u.rt * kTM + half * kHM;
          // Each GO call names a message whose flags ask for a rescale (PV of the
          // message before it has completed), or -1 at the unit's end. Bounded:
          // there are at most n_msgs calls plus the last.
          bool ok = true;
          for (int call = 0; call <= u.n_msgs; ++call) {
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar(B_GO), gcall & 1))) {
              ok = false;
              break;
            }
            ++gcall;
            const int jj = *reinterpret_cast<volatile const int32_t*>(smem + O_GO);
            if (jj < 0) break;
            const int mb = (gb + jj) % kMsgSlots;
            const unsigned char* msg = smem + O_MSG + mb * kMsgStride;
            const uint4 fl = *reinterpret_cast<const uint4*>(msg + kPBytes + kHM * 4);
            const uint32_t mine = qd == 0 ? fl.x : qd == 1 ? fl.y : qd == 2 ? fl.z : fl.w;
            if (mine) {
              const float f = reinterpret_cast<const float*>(msg + kPBytes)[r];
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
            if (lane == 0) {
              if (rank == 2) mbar_arrive(oready);
              else mbar_arrive_cluster(oready);
            }
          }
          // ---- epilogue: O / l -------------------------------------------------
          const int fb = kq & 1;
          const int ml = gb + u.n_msgs - 1;
          ok = __all_sync(0xffffffffu,
                          ok && mbar_wait_cluster(bar(B_FIN_FULL + fb), (kq >> 1) & 1) &&
                              mbar_wait_cluster(bar(B_PV_DONE + ml % kMsgSlots),
                                                (ml / kMsgSlots) & 1));
          if (ok) {
            tc_fence_after();
            const float inv_l = reinterpret_cast<const float*>(smem + O_FIN + fb * kFinBytes)[r];
            // the buffer's next 1/l (two units on) completes its next phase
            if (warp == 2 && lane == 0) mbar_expect_tx(bar(B_FIN_FULL + fb), kFinBytes);
            // Rows go out by TMA stores of 32 rows x 64 dims (two staging boxes
            // per warp, in the 128-byte swizzle) when all 32 rows of the warp
            // exist; a warp that straddles the end of the sequence's rows
            // writes its rows one by one.
            const int lr0 = u.rt * kTM + half * kHM + qd * 32;
            const bool boxed = lr0 + 32 <= QH;
            const bool last_unit = i == n_mine - 1;
            const long long orow = p.n_split == 1 ? 0 : (long long)u.sp * total_rows;
            const int y0 = (int)(orow + row0 + qd * 32);
            __nv_bfloat16* dst_row =
                (p.n_split == 1 ? p.out : p.part_o) + (orow + row0 + r) * (long long)kC;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {  // 128 columns (dims) per TMEM request
              uint32_t ov[128];
              tmem_ld128(t_lane + 128 * c, ov);
              tmem_ld_wait();
              if (c == 3) {
                // both CTAs' O has been read: the next unit's first PV may start
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                  if (rank == 2) mbar_arrive(epi_done + 8 * fb);
                  else mbar_arrive_cluster(epi_done + 8 * fb);
                }
              }
              if (boxed) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int box = 2 * c + h;
                  // The cluster's last unit has the whole value ring to itself
                  // (no value tile follows): each box gets its own staging, so
                  // no store waits for another. Otherwise two boxes per warp in
                  // value stage 2, each reused once the store two back has
                  // read it.
                  const uint32_t bx = last_unit
                                          ? sbase + O_RING + ((uint32_t)qd * 8 + box) * kOutBox
                                          : box_w + (uint32_t)(box & 1) * kOutBox;
                  if (!last_unit && box >= 2) {
                    if (lane == 0) bulk_wait_read1();
                    __syncwarp();
                  }
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    const uint32_t* w = ov + 64 * h + 8 * q;
                    const uint32_t addr = bx + (uint32_t)lane * 128 + ((uint32_t)(q ^ (lane & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "r"(pack_bf16(__uint_as_float(w[0]) * inv_l, __uint_as_float(w[1]) * inv_l)),
                                 "r"(pack_bf16(__uint_as_float(w[2]) * inv_l, __uint_as_float(w[3]) * inv_l)),
                                 "r"(pack_bf16(__uint_as_float(w[4]) * inv_l, __uint_as_float(w[5]) * inv_l)),
                                 "r"(pack_bf16(__uint_as_float(w[6]) * inv_l, __uint_as_float(w[7]) * inv_l))
                                 : "memory");
                  }
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (lane == 0) {
                    if (DDT_GUARD((long long)y0 + 32 <= (p.n_split == 1 ? 1 : p.n_split) * total_rows,
                                  105, p.status + u.b))
                      tma_store_2d(&tm_o, bx, 64 * box, y0);
                    bulk_commit();
                  }
                }
              } else if (row_ok && DDT_GUARD(row0 + r < total_rows, 106, p.status + u.b)) {
                uint4* dst = reinterpret_cast<uint4*>(dst_row + 128 * c);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                  dst[q] = make_uint4(pack_bf16(__uint_as_float(ov[8 * q + 0]) * inv_l,
                                                __uint_as_float(ov[8 * q + 1]) * inv_l),
                                      pack_bf16(__uint_as_float(ov[8 * q + 2]) * inv_l,
                                                __uint_as_float(ov[8 * q + 3]) * inv_l),
                                      pack_bf16(__uint_as_float(ov[8 * q + 4]) * inv_l,
                                                __uint_as_float(ov[8 * q + 5]) * inv_l),
                                      pack_bf16(__uint_as_float(ov[8 * q + 6]) * inv_l,
                                                __uint_as_float(ov[8 * q + 7]) * inv_l));
              }
            }
            if (lane == 0) {
              mbar_arrive_cluster(fin_free + 8 * fb);  // this buffer's 1/l has been read
              bulk_wait_read0();
              mbar_arrive(bar(B_OUT_FREE));            // the staging may take value tiles
            }
          }
          if (!ok) {
            failed = true;
            break;
          }
          gb += u.n_msgs;
          ++kq;
        }
        if (lane == 0) release_unit(i);
      }
    } else if (warp == 6 && rank == 2) {
      // ---------------- the fused tree build --------------------------------
      // One build per unit that walks tree tiles; its ancestor words go to both
      // S-CTAs by 16-byte asynchronous stores from registers (so the build's
      // scratch is free at once), into the buffer of the unit's parity, once
      // the unit two back (the buffer's last user) has ended.
      int kq = 0;
      for (int i = 0; !failed; ++i) {
        Unit u;
        const int t = take_unit(i, u);
        if (t == 0) break;
        if (t < 0) {
          failed = true;
          break;
        }
        if (u.nt == 0) {
          if (u.designated) {  // the tree of a sequence that is not attended is still built
            bool bad = false;
            const int n = fused_build(p.tf, u.b, smem + O_BUILD, &bad);
            fused_write(p, u.b, smem + O_BUILD, n, bad);
          }
        } else {
          if (u.builds) {
            const int vb = kq & 1;
            if (kq >= 2 &&
                !__all_sync(0xffffffffu,
                            mbar_wait_cluster(bar(B_EPI_DONE + vb), ((kq - 2) >> 1) & 1))) {
              failed = true;
              break;
            }
            bool bad = false;
            const int n = fused_build(p.tf, u.b, smem + O_BUILD, &bad);
            __syncwarp();
            const uint4* anc =
                reinterpret_cast<const uint4*>(smem + O_BUILD + offsetof(tb::Smem, anc));
            for (uint32_t s = 0; s < 2; ++s) {
              const uint32_t dst = map_peer(sbase + S_VIS + vb * kVisBuf, s);
              const uint32_t tb_bar = map_peer(bar(B_TREE + vb), s);
              for (int k = lane; k < p.Q; k += 32) {
                const uint4 w = anc[k];
                st_async_v4(dst + 16 * k, w.x, w.y, w.z, w.w, tb_bar);
              }
            }
            if (u.designated) fused_write(p, u.b, smem + O_BUILD, n, bad);
          }
          ++kq;
        }
        if (lane == 0) release_unit(i);
      }
    }
  }

  if (failed) {
    // every sequence of the cluster's units is reported (a wait that gave up
    // may have cut any of them short)
    for (int i = 0;; ++i) {
      const long long uid = unit_id(cl, G, i);
      if (uid >= U) break;
      int b, rt, sp;
      unit_coords(p, order, uid, &b, &rt, &sp);
      atomicOr(p.status + b, DDT_ST_TIMEOUT);
    }
  }
  __syncthreads();
  cluster_sync();  // every pair MMA, copy and remote arrive of the cluster has completed
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  cluster_sync();
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

// Keys: the cache as {64 dims, rows, 9 chunks} (strides: row, 128 B); a box of
// {64, 64, kGroupChunks} at chunk c lands as that many 64-key x 128-byte
// swizzled chunks (8 KB each); a 64-key half of an S tile is kKGroups such
// requests.
// Values: the c_kv part as {64 dims, rows, 4 chunks, 2 halves} (strides: row,
// 128 B, 512 B); a box of {64, 64, 2, 2} at chunk 2h holds dims
// [128h, 128h + 128) and [256 + 128h, 256 + 128h + 128) as four 8 KB chunks.
// Queries: 128 rows per box; q_lat in two boxes of four 64-dim chunks each.
bool encode_maps(CUtensorMap* mk, CUtensorMap* mv, CUtensorMap* ml, CUtensorMap* mp,
                 CUtensorMap* mo, const void* kv, uint64_t kv_rows, const void* q_lat,
                 const void* q_pe, uint64_t q_rows, void* o, uint64_t o_rows) {
  auto fn = encoder();
  if (fn == nullptr) return false;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  const auto oob = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE;
  const auto il = CU_TENSOR_MAP_INTERLEAVE_NONE;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint32_t e4[4] = {1, 1, 1, 1};
  {
    cuuint64_t dims[3] = {64, kv_rows, (cuuint64_t)kChunks};
    cuuint64_t str[2] = {(cuuint64_t)(kC + kR) * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kBK, (cuuint32_t)kGroupChunks};  // a group of chunks
    if (fn(mk, bf, 3, const_cast<void*>(kv), dims, str, box, e4, il, sw, l2, oob) != CUDA_SUCCESS)
      return false;
  }
  {
    cuuint64_t dims[4] = {64, kv_rows, 4, 2};
    cuuint64_t str[3] = {(cuuint64_t)(kC + kR) * 2, 128, 512};
    cuuint32_t box[4] = {64, (cuuint32_t)kBK, 2, 2};
    if (fn(mv, bf, 4, const_cast<void*>(kv), dims, str, box, e4, il, sw, l2, oob) != CUDA_SUCCESS)
      return false;
  }
  {
    cuuint64_t dims[3] = {64, q_rows, (cuuint64_t)(kC / 64)};
    cuuint64_t str[2] = {(cuuint64_t)kC * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kHM, (cuuint32_t)(kC / 128)};  // half the chunks
    if (fn(ml, bf, 3, const_cast<void*>(q_lat), dims, str, box, e4, il, sw, l2, oob) !=
        CUDA_SUCCESS)
      return false;
  }
  {
    cuuint64_t dp[2] = {64, q_rows};
    cuuint64_t spe[1] = {(cuuint64_t)kR * 2};
    cuuint32_t bp[2] = {64, (cuuint32_t)kHM};
    if (fn(mp, bf, 2, const_cast<void*>(q_pe), dp, spe, bp, e4, il, sw, l2, oob) != CUDA_SUCCESS)
      return false;
  }
  // Output (or split-KV partials): rows of 512 dims; a box of {64, 32} is one
  // 64-dim column block of a warp's 32 rows, staged in the 128-byte swizzle.
  cuuint64_t dn[2] = {(cuuint64_t)kC, o_rows};
  cuuint64_t sn[1] = {(cuuint64_t)kC * 2};
  cuuint32_t bn[2] = {64, 32};
  return fn(mo, bf, 2, o, dn, sn, bn, e4, il, sw, l2, oob) == CUDA_SUCCESS;
}

}  // namespace

int verify_attn_pair_clusters_per_wave() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] != 0) return cached[dev];
  static int smem_set[64] = {};
  if (ensure_smem_limit(k_verify_attn_pair, (int)kSmemBytes, smem_set) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * 64, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 4;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_verify_attn_pair, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cached[dev] = n;
  return n;
}

cudaError_t launch_verify_attn_pair(const ddt_attn_dims& d, int n_split, const void* q_lat,
                                    const void* q_pe, const void* kv, const int32_t* block_table,
                                    const int32_t* prefix_len, const uint64_t* vis_bits, void* out,
                                    float* lse, int32_t* status, __nv_bfloat16* part_o,
                                    float* part_lse, cudaStream_t stream, const TreeFuse* fuse) {
  const long long QH = (long long)d.Q * d.H;
  const long long rows = (long long)d.B * QH;
  if (d.kv_rows < 1 || rows > 0x7fffffffLL || d.kv_rows > 0x7fffffffLL || n_split < 1 ||
      (long long)n_split * rows > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  CUtensorMap tm_k, tm_v, tm_ql, tm_qp, tm_o;
  void* o = n_split == 1 ? out : static_cast<void*>(part_o);
  if (!encode_maps(&tm_k, &tm_v, &tm_ql, &tm_qp, &tm_o, kv, (uint64_t)d.kv_rows, q_lat, q_pe,
                   (uint64_t)rows, o, (uint64_t)(rows * n_split)))
    return cudaErrorInvalidValue;
  Params p;
  p.B = d.B; p.Q = d.Q; p.H = d.H;
  p.page_size = d.page_size; p.max_pages = d.max_pages; p.kv_rows = d.kv_rows;
  p.scale_log2 = d.scale * 1.4426950408889634f;
  p.n_rt = (int)((QH + kTM - 1) / kTM);
  p.n_split = n_split;
  p.longest_first = (d.B > 1 && d.B <= kLongestFirstMax) ? 1 : 0;
  p.block_table = block_table; p.prefix_len = prefix_len;
  p.vis_bits = reinterpret_cast<const unsigned long long*>(vis_bits);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse; p.status = status;
  p.part_o = part_o; p.part_lse = part_lse;
  p.fuse = fuse != nullptr ? 1 : 0;
  p.tf = fuse != nullptr ? *fuse : TreeFuse{};
  static int smem_set[64] = {};
  cudaError_t e = ensure_smem_limit(k_verify_attn_pair, (int)kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  // at most as many clusters as are resident at once; each walks its list of
  // units. DDT_PAIR_CLUSTERS (a positive count) sets the number of clusters
  // instead (at most one per unit): a small launch can then run many units per
  // cluster, or a large one one unit per cluster.
  const long long units = (long long)d.B * p.n_rt * n_split;
  long long cap = verify_attn_pair_clusters_per_wave();
  const char* env = getenv("DDT_PAIR_CLUSTERS");
  if (env != nullptr && atoll(env) > 0) cap = atoll(env);
  const long long clusters = cap > 0 && units > cap ? cap : units;
  k_verify_attn_pair<<<(unsigned)(clusters * 4), kThreads, kSmemBytes, stream>>>(
      tm_k, tm_v, tm_ql, tm_qp, tm_o, p);
  return cudaGetLastError();
}

}  // namespace ddt
