/*
 * cpattn.h - C ABI of libcpattn.so: context-parallel causal attention run as a
 * Q-KV task graph on one GB300 GPU (sm_103a).
 *
 * The method, in the words of the pages it follows:
 *  - "Context Parallelism (CP)" (llm-infra-atlas, parallel/04_cp), §2.1: the
 *    query sequence is cut into Q blocks and the key/value sequence into KV
 *    segments; every (Q block, KV segment) pair that the mask does not empty
 *    is an edge of a bipartite task graph, and each edge is one
 *    TileAttention(Q_i, K_j, V_j, M_ij) that yields a partial state
 *    (O_ij, L_ij): O normalised inside the segment, L the row log-sum-exp of
 *    the masked Q_i K_j^T / sqrt(d).
 *  - same page, §2.2: partial states are merged by
 *    L_i = log sum_j exp L_ij,  O_i = sum_j exp(L_ij - L_i) O_ij.
 *  - "04 · Megatron-LM 实现" (llm-infra-atlas, 04_cp/04_megatron_cp_integration),
 *    §1.1 and §1.2: the zigzag split (rank r keeps chunks r and 2cp-1-r of
 *    2cp equal chunks) and its per-sub-sequence form for packed (THD) input.
 *  - "上下文并行：一条序列跨卡，仍算同一个目标" (glenzli.com, context-parallel),
 *    01 and 02: the online recurrence (m, l, a) inside a tile, and the backward
 *    replay from the full-row LSE with dK/dV summed at the key owner.
 *  - "Sequence Parallelism + Ring Attention" (naphjohn LLM-blog), §2: ranks
 *    keep their queries and receive the K/V blocks in ring order.
 * The cp "ranks" are logical: all of them run on one GPU, in ring order, with
 * no collective.
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is DEVICE memory owned by the caller.  The library
 *    never allocates or frees device memory; scratch space is the caller's
 *    workspace (ws, ws_bytes).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on that stream and returns; the
 *    status reports host-side validation and launch errors.  Faults detected
 *    on the device (a bounded wait that ran out) are reported later through
 *    cp_get_device_error().
 *  - Layouts are contiguous, row-major:
 *      BSHD: q, o, dout, dq  [batch][seqlen][heads_q][head_dim]
 *            k, v, dk, dv    [batch][seqlen][heads_kv][head_dim]
 *      THD (cu_seqlens given, batch = 1): the same with seqlen = T.
 *      lse                   [batch][seqlen][heads_q], float32, natural log.
 *    Element type of q/k/v/o/dout/dq/dk/dv: desc->dtype (float32 or bf16).
 *  - Token order: CP_ORDER_ORIGINAL (the sequence as written) or
 *    CP_ORDER_RANK_LOCAL (rank 0's tokens, then rank 1's, ... each rank in the
 *    order of cp_partition_indices), applying to every token-indexed tensor of
 *    a call.
 *  - Grouped heads: q-head h reads kv-head h / (heads_q / heads_kv).
 *  - Attention kernels (cp_tile_attn_fwd, cp_ring_attn_fwd, cp_ring_attn_bwd,
 *    cp_ring_attn_fwd_static_ws) are fixed by the element type: float32 runs
 *    on CUDA-core FFMA kernels (float32 arithmetic, head_dim 64 or 128), bf16
 *    on the tcgen05 tensor-core kernels, built for head_dim 128 only.  bf16
 *    with another head_dim, or a driver that does not export the tensor-map
 *    encoder the tcgen05 kernels need, returns CP_ERR_UNSUPPORTED; no call
 *    switches to another kernel class.  The token gathers and the partition
 *    take both element types at head_dim 64 and 128.
 *  - Status codes are the cp_status values below; no call aborts the process.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1, /* null pointer, bad size, bad cu_seqlens        */
  CP_ERR_ALIGNMENT = -2,   /* a length is not a multiple of 2*cp (striped: cp) */
  CP_ERR_UNSUPPORTED = -3, /* head_dim, dtype or head grouping not built
                              (bf16 attention: head_dim 128 only), or
                              batch * seqlen >= 2^31 token rows           */
  CP_ERR_WORKSPACE = -4,   /* ws too small (see cp_ring_attn_workspace_bytes) */
  CP_ERR_CUDA = -5,        /* a CUDA runtime call failed                   */
  CP_ERR_TIMEOUT = -6      /* a device-side bounded wait ran out           */
} cp_status;

typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype;

typedef enum { CP_ORDER_ORIGINAL = 0, CP_ORDER_RANK_LOCAL = 1 } cp_order;

/* How a sequence (each packed sub-sequence) is split over the cp ranks. */
typedef enum {
  CP_PARTITION_ZIGZAG = 0,  /* 2cp chunks, rank r holds chunks r and 2cp-1-r
                               ("04 · Megatron-LM 实现" §1.1, §1.2)          */
  CP_PARTITION_STRIPED = 1  /* interleaved: token i on rank i mod cp
                               ("Sequence Parallelism + Ring Attention" §5);
                               lengths a multiple of cp, and the token tensors
                               of the ring entry points in rank-local order  */
} cp_partition_scheme;

/* Problem description.  Sizes are in elements. */
typedef struct {
  int32_t batch;       /* BSHD batch; must be 1 for THD                      */
  int32_t heads_q;     /* H                                                  */
  int32_t heads_kv;    /* Hkv, divides H                                     */
  int32_t head_dim;    /* d: 64 or 128                                       */
  int32_t cp;          /* logical context-parallel ranks, >= 1               */
  int32_t causal;      /* 1: causal by original position; 0: full (THD still
                          block-diagonal)                                    */
  int64_t seqlen;      /* BSHD: tokens per batch entry; THD: total tokens T  */
  const int32_t* cu_seqlens_host; /* THD boundaries, HOST memory, [n_seqs+1],
                          cu[0] = 0, cu[n_seqs] = T; NULL for BSHD          */
  const int32_t* cu_seqlens_dev;  /* the same array in DEVICE memory (used by
                          cp_partition_indices); NULL for BSHD             */
  int32_t n_seqs;      /* number of packed sub-sequences (THD), else 0      */
  cp_dtype dtype;      /* element type of the token tensors                 */
  cp_order order;      /* token order of the token tensors                  */
  float softmax_scale; /* 0 -> 1/sqrt(head_dim)                              */
  cp_partition_scheme partition; /* CP_PARTITION_ZIGZAG (0) or _STRIPED     */
  int32_t window;      /* sliding-window width W ("Context Parallelism (CP)"
                          §2.1: a sparser edge set); 0: none.  W > 0 (causal
                          only): the query at position i sees the keys at
                          positions i-W+1 .. i of its (sub-)sequence        */
  /* Hybrid CP ("04 · Megatron-LM 实现" §7, one round of cp_hybrid_schedule;
     THD, zigzag split): sub-sequence k is split by the zigzag rule with
     cp = seq_cp[k] over ranks seq_rank0[k] .. seq_rank0[k] + seq_cp[k] - 1
     (seq_cp[k] a power of two <= cp, seq_rank0[k] a multiple of it), and
     rank r's stream holds, sub-sequence by sub-sequence, the parts of the
     sub-sequences whose group contains r (ranks of different lengths).
     NULL: every sub-sequence spans all cp ranks.                           */
  const int32_t* seq_cp_host;    /* [n_seqs], HOST memory                    */
  const int32_t* seq_rank0_host; /* [n_seqs], HOST memory                    */
  const int32_t* seq_cp_dev;     /* the same arrays in DEVICE memory (used by */
  const int32_t* seq_rank0_dev;  /* cp_partition_indices)                     */
} cp_attn_desc;

/* Human-readable name of a status code (static string). */
const char* cp_status_string(cp_status status);

/* Validate a descriptor without touching the GPU (host logic only).
 * Checks: sizes positive, H % Hkv == 0, d in {64, 128}, batch == 1 for THD,
 * cu_seqlens_host non-decreasing from 0 to T, every sub-sequence length (and
 * the BSHD seqlen) a multiple of 2*cp ("04 · Megatron-LM 实现" §1.1: the
 * sequence length must be divisible by 2*cp); under CP_PARTITION_STRIPED a
 * multiple of cp and order CP_ORDER_RANK_LOCAL (a rank's tokens are strided
 * in the original order), else CP_ERR_UNSUPPORTED.  window: 0 <= W < 2^30
 * (CP_ERR_INVALID_ARG), and W > 0 needs causal = 1 (CP_ERR_UNSUPPORTED).
 * Hybrid CP (seq_cp_host set): THD, zigzag, seq_rank0_host set, every
 * seq_cp[k] a power of two <= cp and seq_rank0[k] a multiple of it with
 * seq_rank0[k] + seq_cp[k] <= cp (else CP_ERR_INVALID_ARG), every length a
 * multiple of 2 * seq_cp[k] (else CP_ERR_ALIGNMENT). */
cp_status cp_validate_desc(const cp_attn_desc* desc);

/* Zigzag / packed partition ("04 · Megatron-LM 实现" §1.1 and §1.2; "Context
 * Parallelism (CP)" §4) or striped partition ("Sequence Parallelism + Ring
 * Attention" §5), as desc->partition says.
 *  idx      [cp][L/cp] int32, device, written: idx[r][t] = original token index
 *           (within one batch entry) held at slot t of rank r.  L = seqlen.
 *           Zigzag BSHD: chunk r then chunk 2cp-1-r of 2cp chunks of L/(2cp)
 *           tokens.  Zigzag THD: for every sub-sequence k in order, its chunk r
 *           then its chunk 2cp-1-r (chunk length len_k / (2cp)).
 *           Striped: for every sub-sequence k (BSHD: the one sequence) in
 *           order, its tokens r, r + cp, r + 2cp, ... (len_k / cp of them).
 *           Hybrid CP: rank r's stream (see cp_attn_desc), ranks in order;
 *           rank r's slice of sub-sequence k is its chunk o = r - seq_rank0[k]
 *           then chunk 2 seq_cp[k] - 1 - o of len_k / (2 seq_cp[k]) tokens.
 *  local_cu [n_seqs+1] int32, device, optional (NULL): boundaries of the
 *           sub-sequences inside one rank's local stream (cu / cp; identical
 *           for every rank).  THD only.  Hybrid CP: [cp][n_seqs+1], REQUIRED:
 *           local_cu[r][k] = the idx slot where rank r's slice of
 *           sub-sequence k starts (empty when r is not in k's group),
 *           local_cu[r][n_seqs] = the end of rank r's stream.
 * Uses desc->cu_seqlens_dev on the device and desc->cu_seqlens_host for
 * validation.  Errors: CP_ERR_ALIGNMENT when a length is not a multiple of
 * 2*cp (striped: cp); CP_ERR_INVALID_ARG for null idx or bad cu_seqlens. */
cp_status cp_partition_indices(const cp_attn_desc* desc, int32_t* idx, int32_t* local_cu,
                               void* stream);

/* Token gather along the sequence (the index_select of "04 · Megatron-LM 实现"
 * §1.1/§1.2) applied to a [batch][seqlen][heads][head_dim] tensor of
 * desc->dtype.  inverse = 0: dst[b][t] = src[b][idx[t]] (original -> rank
 * local); inverse = 1: dst[b][idx[t]] = src[b][t] (rank local -> original).
 * idx is the [cp][seqlen/cp] array of cp_partition_indices.  src and dst must
 * not overlap. */
cp_status cp_permute_tokens(const cp_attn_desc* desc, const int32_t* idx, int32_t heads,
                            const void* src, void* dst, int32_t inverse, void* stream);

/* Per-token metadata of the rank-local order ("04 · Megatron-LM 实现" §1.2:
 * each packed sub-sequence keeps its own positions, counted from 0):
 *  seq_pos [seqlen][2] int32, device, written: for slot t, the index k of the
 *          sub-sequence holding token idx[t] and that token's position in it
 *          (BSHD: k = 0 and the position in the sequence).
 * idx is the array of cp_partition_indices (any split); THD reads
 * desc->cu_seqlens_dev.  Errors: validation errors, CP_ERR_INVALID_ARG for
 * null pointers. */
cp_status cp_token_seq_pos(const cp_attn_desc* desc, const int32_t* idx, int32_t* seq_pos, void* stream);

/* cp_permute_tokens with the rotary position embedding fused in ("04 ·
 * Megatron-LM 实现" §5: the positions must be split by the same zigzag as the
 * tokens; position_ids travel with the tokens).  For a [batch][seqlen][heads]
 * [head_dim] tensor of desc->dtype, pos = the position of token idx[t] in its
 * sequence (BSHD: idx[t]; THD: idx[t] minus the start of its sub-sequence in
 * desc->cu_seqlens_dev), theta_i = pos * rope_base^(-2i/head_dim), i <
 * head_dim/2, and R rotates each pair (x_i, x_{i+head_dim/2}) (the
 * rotate-half pairing) by theta_i:
 *   inverse = 0: dst[b][t] = R(pos) src[b][idx[t]]        (original -> rank local)
 *   inverse = 1: dst[b][idx[t]] = R(pos)^T src[b][t]      (rank local -> original;
 *                the transpose, as for a gradient)
 * Angles are formed and reduced to [-pi, pi] in float64, rotated in float32.
 * Errors: CP_ERR_INVALID_ARG for null pointers, src == dst, heads < 1 or
 * rope_base <= 0; head_dim other than 64/128 is rejected by validation. */
cp_status cp_permute_rope(const cp_attn_desc* desc, const int32_t* idx, int32_t heads, float rope_base,
                          const void* src, void* dst, int32_t inverse, void* stream);

/* One TileAttention edge ("Context Parallelism (CP)" §2.1, A_ij):
 * queries  rows [q_row0, q_row0 + q_len)  of every batch entry of q,
 * keys     rows [kv_row0, kv_row0 + kv_len) of k and v.
 * q_pos0 / kv_pos0 are the ORIGINAL positions of the first row of each range
 * (rows are consecutive positions): with desc->causal, key j is visible to
 * query i iff kv_pos0 + j <= q_pos0 + i, and with desc->window = W > 0 also
 * q_pos0 + i - (kv_pos0 + j) < W.  Both ranges must lie in one sequence (one
 * batch entry, or one packed sub-sequence).
 * Output partial state, float32, device:
 *   o_part   [batch][q_len][heads_q][head_dim]: output normalised over the
 *            visible keys of this segment (0 for a row that sees none);
 *   lse_part [batch][q_len][heads_q]: natural-log LSE of the scaled masked
 *            scores (-inf for a row that sees no key).
 * Errors: CP_ERR_INVALID_ARG if a range leaves the tensor or a length is < 0. */
cp_status cp_tile_attn_fwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           int64_t q_row0, int64_t q_pos0, int64_t q_len, int64_t kv_row0,
                           int64_t kv_pos0, int64_t kv_len, float* o_part, float* lse_part,
                           void* stream);

/* The LSE merge of n_parts partial states ("Context Parallelism (CP)" §2.2):
 *   o_parts   [n_parts][rows][heads][head_dim] float32, device
 *   lse_parts [n_parts][rows][heads]           float32, device
 *   o_out     [rows][heads][head_dim] of out_dtype (float32 or bf16, rounded
 *             to nearest even), lse_out [rows][heads] float32 (may be NULL).
 * L = log sum_j exp L_j (max-shifted), O = sum_j exp(L_j - L) O_j.  Partials
 * with L = -inf weigh 0; if all are -inf the row is O = 0, L = -inf.
 * head_dim must be 64 or 128; n_parts >= 1. */
cp_status cp_merge_partials(int32_t n_parts, int64_t rows, int32_t heads, int32_t head_dim,
                            const float* o_parts, const float* lse_parts, void* o_out,
                            cp_dtype out_dtype, float* lse_out, void* stream);

/* Bytes of workspace cp_ring_attn_fwd (backward = 0) or cp_ring_attn_bwd
 * (backward = 1) needs for this descriptor; 0 if the descriptor is invalid
 * or names an attention shape that is not built (bf16 with head_dim != 128).
 * The workspace must be 256-byte aligned. */
size_t cp_ring_attn_workspace_bytes(const cp_attn_desc* desc, int32_t backward);

/* Context-parallel forward over the whole task graph.
 * For every logical rank r, ring step t = 0..cp-1 (key owner s = (r - t) mod cp,
 * "Sequence Parallelism + Ring Attention" §2), every Q chunk of r and the two
 * KV chunks of s form one edge when some query sees some key; each edge runs
 * TileAttention into a float32 partial state in ws, and the partials of each
 * query row are merged (§2.2 of "Context Parallelism (CP)") into
 *   o   (layout of q, desc->dtype)  and  lse ([batch][seqlen][heads_q] f32).
 * Inputs and outputs are in desc->order.  ws: device, at least
 * cp_ring_attn_workspace_bytes(desc, 0) bytes, 256-byte aligned; its contents
 * need no initialisation and are clobbered.  Calls that share a workspace must
 * not overlap on the GPU.  A descriptor with no tokens (seqlen 0) returns
 * CP_OK at once without reading any pointer; empty sub-sequences of a packed
 * batch own no token and no edge. */
cp_status cp_ring_attn_fwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Context-parallel backward ("上下文并行" 01 BACKWARD/REPLAY and
 * GRADIENT/RETURN, 02 second aligned equations).  Rebuilds the probabilities
 * of every edge from the merged row LSE (P = exp(S - lse)), uses
 * D_i = <dO_i, O_i>, and writes
 *   dq (layout of q), dk, dv (layout of k); dK/dV contributions of every query
 *   rank are summed at the key owner, grouped heads summed into their kv-head.
 * o and lse are cp_ring_attn_fwd's outputs for the same inputs; dout has the
 * layout of q.  ws: at least cp_ring_attn_workspace_bytes(desc, 1) bytes,
 * 256-byte aligned; its contents need no initialisation and are clobbered.
 * For bf16 with head_dim 128 the dq contributions of the key owners are added
 * into a float32 accumulator in ws by hardware reductions whose order is not
 * fixed, so dq may differ in the last bits between calls; dk and dv are
 * summed in a fixed order.  seqlen 0: CP_OK at once, as for the forward. */
cp_status cp_ring_attn_bwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* ws, size_t ws_bytes, void* stream);

/* cp_ring_attn_fwd without a caller workspace, for callers that cannot
 * allocate device memory (no cudaMalloc allowed or available to them).  The
 * pages have no counterpart: this is a property of this library's interface.
 * The scratch is a static device array of cp_static_ws_capacity() bytes
 * (64 MiB) inside the library; every GPU that loads the library keeps it until
 * the process exits.  Same arguments, layouts and results as
 * cp_ring_attn_fwd, minus ws / ws_bytes.
 *  - Returns CP_ERR_WORKSPACE, launching nothing, when the problem needs more
 *    than the static scratch (cp_ring_attn_workspace_bytes(desc, 0) >
 *    cp_static_ws_capacity()).
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.  The first
 *    call in a context (normally once per device, in its primary context)
 *    looks up the scratch's device address (cudaGetSymbolAddress) with that
 *    context current.  A new context (for instance after cudaDeviceReset)
 *    counts as a first call again: the address is looked up anew, never
 *    reused from the old one.
 *  - Every call on a device shares the one scratch array, which keeps the
 *    last call's contents: calls that overlap on the GPU (different streams,
 *    no ordering between them) race and give wrong results. */
cp_status cp_ring_attn_fwd_static_ws(const cp_attn_desc* desc, const void* q, const void* k,
                                     const void* v, void* o, float* lse, void* stream);

/* Size in bytes of the static scratch of cp_ring_attn_fwd_static_ws. */
size_t cp_static_ws_capacity(void);

/* Waits for `stream`, then reads and clears the library's device error word.
 * Returns CP_OK, or CP_ERR_TIMEOUT if a kernel gave up on a bounded wait since
 * the last call (its outputs are then invalid), or CP_ERR_CUDA. */
cp_status cp_get_device_error(void* stream);

/* Failure-detection check: sets the cycle budget of the tcgen05 kernels'
 * main-loop waits (mbarrier and pacing waits) for launches made after this
 * call, process-wide.  cycles <= 0 restores the default of 4e9 cycles (about
 * two seconds); more than the default returns CP_ERR_INVALID_ARG.  While a
 * shorter budget is set, launches run a separately compiled copy of each
 * tcgen05 kernel (the default copies never read the budget, so the setting
 * costs nothing when unused) whose waits probe their barrier without
 * suspending and give up once `cycles` have passed: a budget of a few cycles
 * makes any wait that is not already complete run out.  The block then
 * raises its abort flag, its
 * other roles leave their loops, its TMA copies and MMAs are drained with the
 * default budget, TMEM is freed, and cp_get_device_error reports
 * CP_ERR_TIMEOUT (the outputs of that call are invalid).  The pages have no
 * counterpart ("04 · Megatron-LM 实现" §7.2 shows only the deadlock a missing
 * barrier participant causes).  Not for production use. */
cp_status cp_debug_set_wait_limit(int64_t cycles);

/* Host-only statistics of the task graph built for a descriptor (no GPU use):
 * out[0] forward work items (Q tile x key owner), out[1] partial-state rows
 * per batch entry, out[2] merge segments (Q chunks), out[3] backward work items
 * (KV tile), out[4] unmasked (query, key) pairs per batch entry and head,
 * out[5] forward key-tile visits (128 x 128 tiles) per batch entry and head.
 * Returns CP_OK or the validation error. */
cp_status cp_ring_plan_stats(const cp_attn_desc* desc, int64_t out[6]);

/* Host-only view of the schedule of the tensor-core backward (no GPU use).
 * *grid: CTAs of the launch; *n_work: work indices, w = (batch entry *
 * heads_kv + kv-head) * (backward work items, out[3] of cp_ring_plan_stats)
 * + item.  CTA c runs work[cta[c]] .. work[cta[c + 1] - 1] in that order;
 * load[c] is its planned cost (query tiles x heads per group + 1 per item).
 * Any output pointer may be null; cta holds *grid + 1 entries, work *n_work,
 * load *grid (query the sizes with null arrays first).  Returns CP_OK or the
 * validation error. */
cp_status cp_ring_bwd_schedule(const cp_attn_desc* desc, int32_t* grid, int64_t* n_work, int32_t* cta,
                               int32_t* work, int64_t* load);

/* Hybrid CP schedule ("04 · Megatron-LM 实现" §7.1, the balanced scheduler;
 * §2.3, aligned power-of-two rank groups).  Host only, no GPU.
 * Assigns every sequence a round, a CP size (power of two) and the first
 * rank of its group, longest sequence first:
 *  - a sequence needs the smallest power of two g of ranks with
 *    len <= g * capacity (max(1, 2^ceil(log2(len / capacity)))); its cost on
 *    g ranks is len^2 / g;
 *  - per round: buckets of about equal cost, one per distinct need (closed
 *    past 1.1x the equal share); a sequence joins the least loaded group of
 *    its size with room for len / g more tokens per rank, else opens a group
 *    on the lowest aligned idle block, else waits for the next round; the
 *    round stops at a bucket step once every rank is busy and the loads are
 *    within 5%; the last placed sequences wait while that cuts the spread
 *    of the busy ranks' loads; groups then double over idle buddy blocks,
 *    most loaded first.
 *  lens     [n] HOST, sequence lengths, each a multiple of 2 * world
 *  world    ranks (a power of two); capacity: tokens per rank per round
 *  round, cp, rank0  [n] HOST, written; n_rounds HOST, written
 * Errors: CP_ERR_INVALID_ARG (null pointers, n < 0, world not a power of two,
 * capacity < 1, a negative length), CP_ERR_ALIGNMENT (a length not a
 * multiple of 2 * world), CP_ERR_UNSUPPORTED (a sequence longer than
 * world * capacity). */
cp_status cp_hybrid_schedule(const int32_t* lens, int32_t n, int32_t world, int64_t capacity,
                             int32_t* round, int32_t* cp, int32_t* rank0, int32_t* n_rounds);

/* Host only: the planner's task-graph tables, for tests and tools.
 *  which 0: forward items of 128 query rows (one per Q tile and streaming
 *           part; the FFMA forward), 1: the same parts in 256-row items (the
 *           tensor-core forward), 2: backward items (one K/V tile and every
 *           query range that sees it), 3: dQ items of the FFMA backward (one
 *           Q tile and every key range it sees), 4: merge segments (no
 *           segs; items [n][8]: output row, rows, first partial row, parts,
 *           partial stride, merge row, 0, 0 - output row r + i merges partial
 *           rows first + e * stride + i, e < parts).
 *  items [n_items][8] int32 (which 0-3): stationary tile row, position,
 *           length, first segment, segment count, partial-state row
 *           (forward), cost, 0;
 *  segs  [n_segs][4] int32: streamed range row, position, length, band
 *           (the sliding-window width in the range's positions; 0 none).
 * Rows index the token tensors (desc->order); positions are those the
 * kernels' masks compare (causal: key position <= query position, and
 * query - key < band when band > 0).  Pass null arrays to read the sizes
 * first.  Errors: validation errors, CP_ERR_INVALID_ARG for a bad `which`. */
cp_status cp_ring_plan_tables(const cp_attn_desc* desc, int32_t which, int64_t* n_items, int64_t* n_segs,
                              int32_t* items, int32_t* segs);

/* Kernel classes reported by cp_profile_read. */
typedef enum {
  CP_K_PARTITION = 0, /* partition index kernel                          */
  CP_K_PERMUTE = 1,   /* token gather                                    */
  CP_K_TILE_FWD = 2,  /* tile-attention forward over all edges           */
  CP_K_MERGE = 3,     /* LSE merge                                       */
  CP_K_DELTA = 4,     /* backward preprocess D = rowsum(dO * O)          */
  CP_K_TILE_BWD = 5,  /* tile-attention backward                         */
  CP_K_CONVERT = 6,   /* float32 accumulator -> output dtype             */
  CP_K_TABLES = 7,    /* task-graph table upload (pinned host -> workspace) */
  CP_K_ROPE = 8,      /* token gather with rotary position embedding     */
  CP_K_COUNT = 9
} cp_kernel_class;

/* Benchmark instrumentation (no effect on results).  With timing on, every
 * kernel the library launches is bracketed by two CUDA events recorded on the
 * stream it runs on.  Launch counts are always kept. */
cp_status cp_profile_enable(int32_t on);

/* Waits for the recorded events, writes per-class total device milliseconds
 * (ms[CP_K_COUNT]) and launch counts (launches[CP_K_COUNT]) since the last
 * read, and resets both.  Either pointer may be NULL. */
cp_status cp_profile_read(double* ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
