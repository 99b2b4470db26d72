/*
 * ddt.h -- C ABI of the GB300 (sm_103a) DDTree verify step.
 *
 * One verify step of draft-tree speculative decoding, as a native engine runs
 * it ("The Checkpoint: Committing a Working Native DDTree Engine", section
 * "The Message": generate_ddtree wires tree_build -> verify_attn ->
 * tree_accept + cache compaction):
 *
 *   A. ddt_tree_build     best-first draft tree from the drafter's per-depth
 *                         top-k log-probs
 *   B. ddt_verify_attn    tree-verify MLA-absorb attention over the latent
 *                         cache, mask [ones over prefix | tree visibility]
 *   C. ddt_tree_accept    greedy walk from the root, bonus token
 *   D. ddt_cache_compact  gather of the accepted-path latents
 *   ddt_step              A -> B -> C+D on one stream
 *
 * Conventions (all entry points):
 *  - Every pointer argument is DEVICE memory owned by the caller, except the
 *    dims/args structs, which are read on the host during the call. The
 *    library keeps no pointer after it returns and allocates no device memory;
 *    scratch space is passed in (size it with the *_workspace_size query).
 *  - Work is enqueued on `stream` and the call returns without synchronising.
 *    Results are ready when the stream reaches them.
 *  - The return value reports problems found on the HOST (bad sizes, null
 *    pointers, unsupported dimensions, launch failures): DDT_OK or a negative
 *    DDT_E* code; nothing was enqueued when it is negative (DDT_ELAUNCH: some
 *    earlier kernels of the same call may have been enqueued).
 *  - Problems in the DATA are found on the device and reported per sequence
 *    in `status` (int32[B]) as DDT_ST_* bits; kernels never trap, every
 *    device loop is bounded and every wait gives up after about a second
 *    (DDT_ST_TIMEOUT). ddt_tree_build and ddt_step overwrite status[b];
 *    ddt_verify_attn, ddt_tree_accept and ddt_cache_compact OR their bits in.
 *  - Integer arrays are int32, row-major, densely packed (strides in the
 *    comments). Nodes of a tree are numbered in the order the builder pops
 *    them: slot 0 is the root, and every node's parent has a lower slot.
 *  - Thread-compatible: calls on different streams may run concurrently. The
 *    library's global state is a per-device cache of device properties, plus
 *    what ddt_verify_attn_noalloc needs: a 32 MiB device array reserved on
 *    every GPU that loads the library, and a per-device cache of its address.
 */
#ifndef DDT_H_
#define DDT_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host return codes ---------------------------------------------------- */
#define DDT_OK 0
#define DDT_EINVAL (-1)       /* invalid argument (null pointer, negative size, ...) */
#define DDT_EUNSUPPORTED (-2) /* valid but outside what this library supports */
#define DDT_ELAUNCH (-3)      /* a CUDA launch or query failed */
#define DDT_EWORKSPACE (-4)   /* workspace missing or smaller than required */

/* ---- per-sequence device status bits ------------------------------------- */
#define DDT_ST_BUDGET_PAD 1  /* tree has fewer than budget+1 nodes; the rest is padding (informational) */
#define DDT_ST_INPUT 2       /* non-finite log-prob, or a token id outside [0, V) */
#define DDT_ST_CYCLE 4       /* accept walk would revisit a node (malformed tree) */
#define DDT_ST_RANGE 8       /* accept path / slot outside the cache; sequence left untouched */
#define DDT_ST_CAPACITY 16   /* prefix_len + q_len exceeds the sequence's cache capacity */
#define DDT_ST_TIMEOUT 32    /* a device-side wait ran past its bound (about 1 s); this sequence's outputs are not valid */
#define DDT_ST_CHECK 64      /* (library built with DDT_CHECKS) a device bounds check failed; the access was skipped or clamped */

/* ---- element types -------------------------------------------------------- */
#define DDT_F32 0  /* float32 inputs and outputs; SIMT fp32 arithmetic (exactness path) */
#define DDT_BF16 1 /* bfloat16 inputs and outputs; tensor cores, fp32 accumulation */

/* Largest supported q_len (= budget + 1); the mask of a query row is
 * W = ceil(q_len / 64) uint64 words. */
#define DDT_MAX_Q 128

/* Shapes of the tree build. B sequences, D draft depths, K candidates per
 * depth, budget draft nodes (q_len = budget + 1 tree slots), vocabulary V. */
typedef struct ddt_tree_dims {
  int32_t B, D, K, budget, V;
} ddt_tree_dims;

/* Shapes of the verify attention.
 *  B sequences, Q = q_len tree queries per sequence, H query heads,
 *  C = kv_lora_rank (latent width), R = rope width; the cache row of a token
 *  is [c_kv (C) | k_pe (R)].
 *  The cache is paged: slot s of sequence b lives in physical row
 *  block_table[b * max_pages + s / page_size] * page_size + s % page_size of a
 *  [kv_rows, C+R] array (a contiguous cache is max_pages = 1 with a page per
 *  sequence). scale multiplies q.k. max_len is a host-side upper bound of
 *  prefix_len[b] + Q over the batch; it only sizes the split of the key range
 *  (and so the workspace), results are correct for any length that fits the
 *  cache. */
typedef struct ddt_attn_dims {
  int32_t B, Q, H, C, R;
  int32_t page_size, max_pages;
  int32_t dtype; /* DDT_F32 or DDT_BF16 */
  int64_t kv_rows;
  float scale;
  int32_t max_len;
} ddt_attn_dims;

/* A. Best-first draft-tree construction.
 * "The Milestone Commit: Cementing a Native DDTree Inference Engine", sections
 * "What the Message Actually Does" (GPU best-first tree builder, double
 * accumulation for parity, ancestor-bitmask visibility, first-child /
 * next-sibling retrieve) and "The Reasoning Behind the Architecture".
 *
 * Node score = sum of the log-probs along its path, accumulated in double
 * (child = parent + (double)logp). Starting from the root (score 0), the best
 * frontier node is popped, then its first child (rank 0, one depth down) and
 * its next sibling (rank+1, same parent) are pushed; order is score
 * descending, then depth ascending, then rank ascending, then parent slot
 * ascending. Construction stops after `budget` pops. Every node at depth d
 * takes its token and log-prob from row d-1 of the drafter's top-k.
 *
 * In:  topk_logp f32[B][D][K] (rank 0 first), topk_ids i32[B][D][K],
 *      root_tok i32[B] (the verified token at slot 0).
 * Out (Q = budget+1, W = ceil(Q/64)):
 *      tokens, parents (root -1), depths (root 0): i32[B][Q];
 *      vis_bits u64[B][Q][W]: bit t of word t/64 of row n is set iff slot t is
 *        n or an ancestor of n;
 *      vis u8[B][Q][Q] (may be NULL): the same mask expanded, 1 = visible;
 *      first_child, next_sibling i32[B][Q] (-1 = none; lowest slot first);
 *      n_nodes i32[B]; status i32[B] (overwritten).
 * Slots n_nodes..Q-1 (only when the candidate tree is smaller than the budget,
 * DDT_ST_BUDGET_PAD) hold token 0, parent -1, depth -1, self-visibility only.
 * A NaN/inf log-prob or an id outside [0, V) sets DDT_ST_INPUT and yields the
 * root alone. Limits: 1 <= B, 1 <= D, 1 <= K, 0 <= budget < DDT_MAX_Q,
 * min(D,budget) * min(K,budget) <= 8192, V >= 1. */
int ddt_tree_build(const ddt_tree_dims* dims, const float* topk_logp, const int32_t* topk_ids,
                   const int32_t* root_tok, int32_t* tokens, int32_t* parents, int32_t* depths,
                   uint64_t* vis_bits, uint8_t* vis, int32_t* first_child, int32_t* next_sibling,
                   int32_t* n_nodes, int32_t* status, cudaStream_t stream);

/* Bytes of scratch ddt_verify_attn needs for these dims (0 = none). */
size_t ddt_verify_attn_workspace_size(const ddt_attn_dims* dims);

/* Query rows per tile (128 or 256) the DDT_BF16 verify attention uses for
 * these dims on the current device: 256-row tiles run on paired SMs (four-CTA
 * clusters) and are taken when padding a sequence's Q*H rows to a multiple of
 * 256 costs at most 1/12 of them; the environment variable
 * DDT_VERIFY_ATTN_ROWS (128 or 256) overrides the choice. Informational (no
 * counterpart on the source pages); 0 for invalid or DDT_F32 dims. */
int ddt_verify_attn_rows_per_tile(const ddt_attn_dims* dims);

/* Number of key ranges each sequence's keys are split into by the DDT_BF16
 * verify attention for these dims on the current device (1: no split and no
 * merge pass; >1: partial results in the workspace, merged by a second
 * kernel). Informational (no counterpart on the source pages); 0 for invalid
 * or DDT_F32 dims. */
int ddt_verify_attn_splits(const ddt_attn_dims* dims);

/* B. Tree-verify MLA-absorb attention.
 * "The Checkpoint: Committing a Working Native DDTree Engine", section "The
 * Message" (attention via the custom verify_attn in absorb form; KV-cache
 * scheme: the tree [verified_id, drafts] sits at cache positions L+depth,
 * prefix = cache length, mask = [ones | visibility], AR = degenerate
 * q_len = 1) and "The Milestone Commit", section "Input Knowledge Required"
 * (MLA latent cache, kv_lora_rank 512 for Kimi K2.6).
 *
 * For sequence b (L = prefix_len[b]), tree query i and head h:
 *   s_j = (q_lat[b,i,h,:] . c_kv[j,:] + q_pe[b,i,h,:] . k_pe[j,:]) * scale
 * over key slots j in [0, L) (always visible) and j = L + t for tree slots t
 * visible from i (bit t of vis_bits[b][i]); p = softmax(s);
 *   out[b,i,h,:] = sum_j p_j c_kv[j,:],  lse[b,i,h] = log sum_j exp(s_j).
 * The caller has already written the tree nodes' latents into slots
 * [L, L+Q) in node (slot) order.
 *
 * q_lat [B][Q][H][C], q_pe [B][Q][H][R], kv_cache [kv_rows][C+R], out
 * [B][Q][H][C]: element type dims->dtype. block_table i32[B][max_pages],
 * prefix_len i32[B], vis_bits u64[B][Q][W]; lse f32[B][Q][H] (may be NULL);
 * status i32[B] (OR-ed). A sequence with prefix_len < 0 or
 * prefix_len + Q > max_pages * page_size gets DDT_ST_CAPACITY, and one with a
 * page of [0, prefix_len + Q) outside the kv_rows of the cache gets
 * DDT_ST_RANGE; either way its output is zero and its lse -inf, and nothing
 * outside its valid pages is read.
 * DDT_BF16 requires C = 512, R = 64 (tcgen05 kernel), scale > 0, page_size a
 * multiple of 64 and 16-byte aligned pointers; DDT_F32 takes any C <= 1024, R <= 256.
 * Both need 1 <= Q <= DDT_MAX_Q. workspace: at least
 * ddt_verify_attn_workspace_size(dims) bytes of device memory (may be NULL
 * when that is 0), 256-byte aligned. */
int ddt_verify_attn(const ddt_attn_dims* dims, const void* q_lat, const void* q_pe,
                    const void* kv_cache, const int32_t* block_table, const int32_t* prefix_len,
                    const uint64_t* vis_bits, void* out, float* lse, int32_t* status,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* B'. The bf16 verify attention of ddt_verify_attn, for callers that cannot
 * allocate device memory. This entry point has no counterpart on the source
 * pages; it exists for code that can hand the library its inputs and outputs
 * but cannot obtain scratch memory (device allocation forbidden or
 * unavailable where it runs, e.g. a plugin given only its I/O buffers, or a
 * loop that must never enter an allocator).
 * Same arguments and results as ddt_verify_attn with dims->dtype == DDT_BF16,
 * minus the workspace: the split-KV scratch comes from a fixed 32 MiB array
 * the library reserves on every GPU that loads it (held until exit). Returns
 * DDT_EWORKSPACE, before enqueuing anything, when these dims need more
 * scratch than that (ddt_verify_attn_workspace_size(dims) > 32 MiB), and
 * DDT_EUNSUPPORTED for DDT_F32. All calls share the array: calls whose GPU
 * work may overlap (several streams or host threads) race and must be
 * serialised by the caller. The first call on a device looks up the array's
 * address with that device current and keeps it (first calls from several host
 * threads at once are safe); make it before any stream capture, and do not
 * use this entry point after a cudaDeviceReset of that device. */
int ddt_verify_attn_noalloc(const ddt_attn_dims* dims, const void* q_lat, const void* q_pe,
                            const void* kv_cache, const int32_t* block_table,
                            const int32_t* prefix_len, const uint64_t* vis_bits, void* out,
                            float* lse, int32_t* status, cudaStream_t stream);

/* C. Greedy tree accept.
 * "The Checkpoint", section "The Message" (tree_accept; DDTree greedy
 * output == AR greedy output) and "The Milestone Commit", section "Mistakes
 * and Incorrect Assumptions" (the walk carries a safety bound since cyclic
 * input crashed it).
 *
 * Start at the root; at most D times, move to the lowest-slot child c of the
 * current node (parents[c] == current) whose token equals
 * target_argmax[current]; stop when there is none. A move to a node already
 * on the path stops the walk with DDT_ST_CYCLE. bonus = target_argmax at the
 * last node.
 * In:  tokens, parents, target_argmax: i32[B][Q] (indexed by tree slot).
 * Out: accept_idx i32[B][D+1] (slot 0 = root, then the accepted slots, -1
 *      after), accept_len i32[B] (accepted drafts, root excluded),
 *      out_tokens i32[B][D+1] (accepted draft tokens, then the bonus, -1
 *      after), bonus i32[B], status i32[B] (OR-ed).
 * Limits: 1 <= Q <= DDT_MAX_Q, D >= 0. */
int ddt_tree_accept(int32_t B, int32_t Q, int32_t D, const int32_t* tokens,
                    const int32_t* parents, const int32_t* target_argmax, int32_t* accept_idx,
                    int32_t* accept_len, int32_t* out_tokens, int32_t* bonus, int32_t* status,
                    cudaStream_t stream);

/* D. Post-verify cache compaction.
 * "The Checkpoint", section "The Message" (cache append + post-verify
 * compaction; after accept, gather the accepted-path latents; gather/copy
 * rows).
 *
 * For d = 1..accept_len[b]: the row at slot L + accept_idx[b][d] is copied to
 * slot L + d (L = prefix_len[b]; the root stays at slot L), with every source
 * row read before any destination row is written. new_len[b] = L + 1 +
 * accept_len[b]. kv_cache is [kv_rows][row_bytes] bytes, paged as in
 * ddt_attn_dims. accept_idx[b][1..accept_len] must be a path from the root
 * (slot 0) in pop order, as ddt_tree_accept writes it: strictly increasing,
 * first entry >= 1 (accept_idx[b][0] is not read). Rows already in place
 * (accept_idx[b][d] == d) are not touched. A sequence whose list is not such
 * a path, whose slots fall outside [0, max_pages * page_size), or whose pages
 * fall outside the kv_rows of the cache, is left untouched, new_len = L,
 * DDT_ST_RANGE.
 * Limits: row_bytes a positive multiple of 16, D <= DDT_MAX_Q - 1. */
int ddt_cache_compact(int32_t B, int32_t D, int32_t row_bytes, int32_t page_size,
                      int32_t max_pages, int64_t kv_rows, void* kv_cache,
                      const int32_t* block_table,
                      const int32_t* prefix_len, const int32_t* accept_idx,
                      const int32_t* accept_len, int32_t* new_len, int32_t* status,
                      cudaStream_t stream);

/* Everything one verify step reads and writes; see the four calls above for
 * each array's meaning and layout. tree.B == attn.B and attn.Q ==
 * tree.budget + 1. target_argmax (i32[B][Q], per tree slot) stands for the
 * target model's argmax after the verify forward; it must be consistent with
 * the tree this step builds (the builder is deterministic). */
typedef struct ddt_step_args {
  ddt_tree_dims tree;
  ddt_attn_dims attn;
  const float* topk_logp;
  const int32_t* topk_ids;
  const int32_t* root_tok;
  const void* q_lat;
  const void* q_pe;
  void* kv_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* target_argmax;
  int32_t* tokens;
  int32_t* parents;
  int32_t* depths;
  uint64_t* vis_bits;
  uint8_t* vis; /* may be NULL */
  int32_t* first_child;
  int32_t* next_sibling;
  int32_t* n_nodes;
  void* out;
  float* lse; /* may be NULL */
  int32_t* accept_idx;
  int32_t* accept_len;
  int32_t* out_tokens;
  int32_t* bonus;
  int32_t* new_len;
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
} ddt_step_args;

/* Bytes of scratch ddt_step needs. */
size_t ddt_step_workspace_size(const ddt_step_args* args);

/* A -> B -> C+D on `stream`: tree build, verify attention, accept and
 * compaction (accept and compaction run fused in one kernel; when B splits
 * the key range, its merge pass runs beside C+D, which needs only the tree
 * and B's finished cache reads). Everything enqueued after ddt_step sees the
 * whole step done. status is overwritten, then OR-ed by every stage. */
int ddt_step(const ddt_step_args* args, cudaStream_t stream);

/* Target-side argmax at every tree slot: the target model's greedy token,
 * the input tree_accept compares the drafted tokens with.
 * "The Checkpoint: Committing a Working Native DDTree Engine", section "The
 * Message" (the target's argmax at each tree node feeds tree_accept).
 *
 * logits: rows x V values, row-major (rows = B * Q tree slots, in the slot
 * order of the tree arrays), dtype DDT_BF16 or DDT_F32, caller-owned device
 * memory. argmax: int32 [rows], caller-owned device memory, written with the
 * index of each row's largest logit: ties go to the lowest index, -0.0 equals
 * +0.0, a NaN counts as larger than every number (the first NaN wins).
 * Rows that start on a 16-byte boundary with V a multiple of 8 (bf16) or 4
 * (f32) are read with vector loads, others element by element; any V >= 1 is
 * accepted. Limits: 1 <= rows <= 2^28 - 1, 1 <= V <= 2^31 - 1. Returns
 * DDT_EINVAL for a null pointer, a size below 1 or an unknown dtype,
 * DDT_EUNSUPPORTED past the limits. Enqueues one kernel on `stream`;
 * allocates nothing. */
int ddt_target_argmax(int64_t rows, int64_t V, int dtype, const void* logits, int32_t* argmax,
                      cudaStream_t stream);

/* Drafter-side per-depth top-K: the K largest logits of every row and their
 * log-probabilities, the input of ddt_tree_build.
 * "The Milestone Commit: Cementing a Native DDTree Inference Engine",
 * section "What the Message Actually Does" (the GPU tree builder consumes the
 * drafter's per-depth top-K log-probs); node score = sum of log-probs along
 * the path.
 *
 * logits: rows x V values, row-major (rows = B * D: sequence, then depth),
 * DDT_BF16 or DDT_F32, caller-owned device memory; finite values and -inf
 * (at least one finite value per row). topk_logp: float [rows, K],
 * topk_ids: int32 [rows, K], caller-owned device memory, written rank 0
 * first: the K largest logits by value (descending), ties to the lower token
 * id, with log-prob = logit - log(sum over the row of exp(logit)), computed
 * in fp32 (an online log-sum-exp; within 1e-5 of the exact value at
 * V = 163840). Rows read with vector loads when 16-byte aligned with V a
 * multiple of 8 (bf16) or 4 (f32). Limits: 1 <= K <= 16, K <= V,
 * 1 <= rows <= 2^28 - 1, V <= 2^31 - 1. Returns DDT_EINVAL for a null
 * pointer, a size below 1 or an unknown dtype, DDT_EUNSUPPORTED past the
 * limits. Enqueues one kernel; allocates nothing. */
int ddt_drafter_topk(int64_t rows, int64_t V, int32_t K, int dtype, const void* logits,
                     float* topk_logp, int32_t* topk_ids, cudaStream_t stream);

/* Rotary embedding of the tree at positions L+depth and append of the tree
 * latents to the paged cache (the step between the target's projections and
 * ddt_verify_attn).
 * "The Checkpoint: Committing a Working Native DDTree Engine", section "The
 * Message" (KV-cache scheme: [verified_id, drafts] processed at positions
 * L+depth, prefix = cache length; the model's cache append before
 * attention); "The Consolidation Point: Validating Generality and Wrapping
 * the MVP", section "The Journey to This Point" (NeoX-style rotary
 * embedding).
 *
 * dims: B, Q, H, C, R, page_size, max_pages, dtype and kv_rows as in
 * ddt_attn_dims (scale and max_len are not used); R even, 2 <= R <= 256,
 * C >= 0, any page_size >= 1. theta: the rotary base (> 0, finite).
 * For sequence b (L = prefix_len[b]) and tree slot t the position is
 * p = L + max(depths[b][t], 0) (padding slots, depth -1, take L); pair i of
 * a rope part, (x_i, x_{i+R/2}), turns by p * theta^(-2i/R):
 *   y_i = x_i cos - x_{i+R/2} sin,  y_{i+R/2} = x_{i+R/2} cos + x_i sin.
 * q_pe_in [B][Q][H][R] -> q_pe_out [B][Q][H][R] (the same pointer rotates in
 * place; otherwise the buffers must not overlap). kv_new [B][Q][C+R] (latent
 * part, then the unrotated rope part) -> cache slot L + t of kv_cache
 * [kv_rows][C+R] (paged through block_table i32[B][max_pages]), latent part
 * copied bit for bit and rope part rotated; kv_new must not overlap the
 * cache. The angles are formed in double and reduced modulo 2*pi before a
 * float sine and cosine, the pairs turn in fp32 and are rounded once to the
 * element type: within 1e-6 * (|x_i| + |x_{i+R/2}|) of the exact rotation
 * before that rounding. A sequence with L < 0 or L + Q > max_pages *
 * page_size gets DDT_ST_CAPACITY, one with a slot of [L, L+Q) on a page
 * outside the kv_rows rows DDT_ST_RANGE (status i32[B], OR-ed); nothing of
 * it is written. All pointers are caller-owned device memory. Limits:
 * 1 <= Q <= DDT_MAX_Q, B * Q <= 2^31 - 1. Returns DDT_EINVAL for a null
 * pointer, a bad size, an odd R or a bad theta, DDT_EUNSUPPORTED past the
 * limits. Enqueues one kernel; allocates nothing. */
int ddt_rope_append(const ddt_attn_dims* dims, double theta, const int32_t* depths,
                    const int32_t* prefix_len, const int32_t* block_table, const void* q_pe_in,
                    void* q_pe_out, const void* kv_new, void* kv_cache, int32_t* status,
                    cudaStream_t stream);

/* ---- multi-step decode loop ------------------------------------------------
 * DDTree greedy decoding of several tokens per sequence, all steps on the
 * device: one CUDA graph whose conditional WHILE node repeats a verify step
 * until every sequence has n_new tokens after its first, or max_steps steps
 * have run.
 * "The Checkpoint: Committing a Working Native DDTree Engine", section "The
 * Message" (generate_ddtree wires tree_build -> verify_attn -> tree_accept +
 * cache compaction with a drafter interface; DDTree greedy == AR greedy; the
 * oracle drafter accepts 8.00 tokens per step, 3 verify steps for 24 tokens).
 *
 * A step: the drafter's logits for depths 1..D -> ddt_drafter_topk ->
 * ddt_tree_build (root = last committed token) -> ddt_rope_append ->
 * ddt_verify_attn -> the target's logits at every tree slot ->
 * ddt_target_argmax -> accept + compaction -> commit (accepted drafts, then
 * the bonus token, which is the next root; the cache length becomes the
 * compacted length).
 * The two model interfaces are synthetic stand-ins: the DRAFTER's logits
 * for depth d are row n - 1 + d of drafter_table[b] (n = tokens committed so
 * far; row g holds the logits for stream position g, clamped to the table),
 * and the TARGET's greedy token at a tree slot is golden[b][n + depth] when
 * the slot's path from the root follows golden[b], else V-1 (and V-1 at
 * padding slots); the target's logits row is 1 there and 0 elsewhere. With
 * such a target, autoregressive greedy decoding yields golden[b] itself.
 * The projections the verify step attends with are fixed inputs (q_lat,
 * q_pe, kv_new), the same every step. */
typedef struct ddt_loop_args {
  ddt_tree_dims tree; /* B, D, K, budget, V */
  ddt_attn_dims attn; /* B, Q = budget + 1, H, C, R, paging, dtype (also of both logits
                         tables), kv_rows, scale; max_len bounds prefix_len0 + n_new +
                         budget + 1 over the batch */
  double theta;       /* rotary base */
  int32_t n_new;      /* tokens to add to each sequence after its first (>= 0) */
  int32_t max_steps;  /* bound on the verify steps (>= 1) */
  int32_t golden_len; /* G >= 2: length of every golden stream and drafter table */
  const int32_t* golden;     /* [B][G] target stream; golden[b][0] is the first token */
  const void* drafter_table; /* [B][G][V] drafter logits per stream position */
  const void* q_lat;         /* [B][Q][H][C] */
  const void* q_pe;          /* [B][Q][H][R], before rotation */
  const void* kv_new;        /* [B][Q][C+R], rope part before rotation */
  void* kv_cache;            /* [kv_rows][C+R], paged by block_table */
  const int32_t* block_table;  /* [B][max_pages] */
  const int32_t* prefix_len0;  /* [B] cache length before the first step */
  int32_t* prefix_len;         /* [B] working cache length; the final length after */
  int32_t* committed;          /* out [B][n_new + 1]: the first token, then the decoded ones */
  int32_t* n_committed;        /* out [B] */
  int32_t* steps;              /* out [B]: verify steps this sequence took */
  int32_t* accepted;           /* out [B][max_steps]: tokens each step committed (before
                                  cutting at n_new), 0 after the last */
  int32_t* status;             /* out [B]: error bits of the step that stopped a sequence */
  void* workspace;             /* ddt_loop_workspace_size bytes, 256-byte aligned */
  size_t workspace_bytes;
} ddt_loop_args;

typedef struct ddt_loop ddt_loop; /* an instantiated loop graph */

/* Bytes of workspace the loop needs (0 for invalid args). */
size_t ddt_loop_workspace_size(const ddt_loop_args* args);

/* Capture the loop body (every step's launches, with these pointers) into a
 * graph and instantiate it. The step's host checks run here: their DDT_E*
 * code is returned and nothing is kept. Device memory is not touched. */
int ddt_loop_create(const ddt_loop_args* args, ddt_loop** loop);

/* Reset the loop state (committed = the first golden token, cache length =
 * prefix_len0, outputs cleared) and run the whole loop on `stream`. May be
 * called repeatedly; calls on the same loop must not overlap. */
int ddt_loop_launch(ddt_loop* loop, cudaStream_t stream);

/* Free the graph (deferred by CUDA until a launch in flight completes). */
int ddt_loop_destroy(ddt_loop* loop);

/* Self-test of the bounded device waits (failure detection; no counterpart on
 * the source pages). Every kernel of this library waits on mbarrier phases
 * with a limit of about one second, after which it records DDT_ST_TIMEOUT for
 * the sequence and leaves instead of hanging. This runs that mechanism alone
 * in one small kernel on `stream`: result (device, int32[3]) receives
 * [0] the status of a wait on a phase nothing completes (DDT_ST_TIMEOUT
 * expected), [1] the status of a wait on a completed phase (0 expected) and
 * [2] how long the first wait lasted in milliseconds. Takes about a second. */
int ddt_wait_selftest(int32_t* result, cudaStream_t stream);

/* Static text for a DDT_E* return code. */
const char* ddt_strerror(int code);

/* Debug-build bounds checks (SURVEY's safety plan; no counterpart on the
 * source pages). A library built with -DDDT_CHECKS (libddt_checks.so) tests
 * every computed global row, page and TMA coordinate before the access it
 * guards; a failing check skips the access (or clamps a TMA coordinate to a
 * valid row, so that no barrier is left waiting), counts the failure, keeps
 * the id of the first failing site, and ORs DDT_ST_CHECK into the sequence's
 * status where the call has one. This reads and resets the counts: it
 * returns 1 in such a library (0 in the release library, whose checks
 * compile to nothing), with n_failed the number of failed checks since the
 * last call and first_site the id of the earliest (file * 100 + site; 0 if
 * none). Synchronises the device. */
int ddt_debug_checks(int* n_failed, int* first_site);

/* The cudaError_t behind the calling thread's most recent DDT_ELAUNCH
 * (0 when there was none), and the CUDA runtime's name for such a value
 * (static text, never NULL). */
int ddt_last_cuda_error(void);
const char* ddt_cuda_error_name(int err);

/* Version of this ABI (increments on any incompatible change). */
int ddt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DDT_H_ */
