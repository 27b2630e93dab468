/*
 * anchorattn.h — C ABI of the GB300 (sm_103a) fused RoPE + AnchorAttention
 * library (libanchorattn.so).
 *
 * The method: "When Precision Meets Position: BFloat16 Breaks Down RoPE in
 * Long-Context Training" (arXiv 2411.13476). Operation references below name
 * the page and its section:
 *   [ARCH §3.4 RoPE]    architecture page, §3.4 "Rotary Positional Embedding
 *                       (RoPE): The Theoretical Promise", Eq. 6 and Eq. 3.
 *   [ARCH §3.4 Index]   architecture page, §3.4 "Document Token Indexing"
 *                       (continuous IDs, Fig. 2 left; reset IDs, Fig. 2 middle).
 *   [ARCH §3.4 Anchor]  architecture page, §3.4 "AnchorAttention: The Shared
 *                       Anchor Design", "Core design" and "Mask construction".
 *   [ARCH §3.2]         architecture page, §3.2 "Big-Picture Architecture":
 *                       RoPE in fp32, cast to bf16, inner products in bf16.
 *   [ARCH §3.4 Diag]    architecture page, §3.4 "Diagnostic Methodology:
 *                       Measuring the Breakdown", Eq. 4 (attention difference)
 *                       and Eq. 5 (first-token logit difference).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned, contiguous, row-major [T, H, D] bf16 (token,
 *    head, channel), 16-byte aligned device pointers. LSE/D-style per-row
 *    values are fp32 [H, T].
 *  - Q and K are passed UN-ROTATED: the library rotates them (RoPE in fp32,
 *    rounded to bf16) once per call in its own kernels; gradients are returned
 *    with respect to the un-rotated inputs (aa_bwd_from_fwd takes the
 *    forward's rotated copies instead of q and k).
 *  - Token 0 is the anchor. cu_doclens (host int32[num_docs + 1]) gives the
 *    document boundaries after it: document k occupies tokens
 *    [cu[k-1], cu[k]), with cu[0] == 1, cu[num_docs] == T, strictly increasing.
 *    In AA_MASK_CAUSAL mode cu_doclens is ignored (may be NULL).
 *  - Every call validates its arguments synchronously and returns a status
 *    without launching anything on failure. Kernel launches are asynchronous
 *    on `stream` (NULL = the legacy default stream); launch failures return
 *    AA_ERR_CUDA. Device-side waits are bounded: a wait that runs out records
 *    an error word that aa_check_device_error() turns into AA_ERR_TIMEOUT.
 *  - aa_fwd / aa_bwd / aa_rope_apply allocate no memory (scratch comes from
 *    caller workspaces sized by aa_*_workspace_bytes). aa_plan allocates the
 *    plan's device metadata; aa_plan_destroy frees it.
 *  - Compute calls may overlap on the GPU when each has its own workspace
 *    (the persistent kernels keep their work counters there); calls with one
 *    plan share its device error word, so aa_check_device_error() reports a
 *    timeout from any of them.
 *  - The compute calls enqueue only stream-ordered work (kernel launches and
 *    asynchronous memsets of their work counters), so a sequence of them may
 *    be captured in a CUDA graph and replayed while the plan, the tensors and
 *    the workspaces it names stay alive. Make one uncaptured call of each
 *    entry point per device first: the first call sets the kernels'
 *    shared-memory attributes (aa_bwd_static_workspace also looks up its
 *    array's address then).
 *  - A thread-local message describing the last failure is available from
 *    aa_last_error().
 */
#ifndef ANCHORATTN_H
#define ANCHORATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* aa_stream_t; /* identical to cudaStream_t */

typedef enum {
  AA_OK = 0,
  AA_ERR_INVALID_ARG = 1,
  AA_ERR_UNSUPPORTED = 2,
  AA_ERR_CUDA = 3,
  AA_ERR_NO_MEMORY = 4,
  AA_ERR_TIMEOUT = 5
} aa_status;

/* Which (query, key) pairs are visible. [ARCH §3.4 Anchor], [ARCH §3.4 Index]
 * CAUSAL:    j <= i over the whole packed sequence (full attention baseline).
 * INTRA_DOC: j <= i and same document; the anchor is a one-token document.
 * ANCHOR:    INTRA_DOC plus key 0 (the anchor) visible to every query; the
 *            anchor query sees only itself. */
typedef enum { AA_MASK_CAUSAL = 0, AA_MASK_INTRA_DOC = 1, AA_MASK_ANCHOR = 2 } aa_mask_mode;

/* Position IDs [ARCH §3.4 Index]. RESET: anchor 0, every document 1..N_k.
 * CONTINUOUS: 0..T-1 across documents. CAUSAL mode always uses 0..T-1. */
typedef enum { AA_POS_RESET = 0, AA_POS_CONTINUOUS = 1 } aa_pos_mode;

/* Pairing of rotated coordinates. ADJACENT = Eq. 6 of [ARCH §3.4 RoPE]
 * (pairs (2p, 2p+1)); HALF pairs (p, p + D/2); NONE disables the rotation. */
typedef enum { AA_ROPE_ADJACENT = 0, AA_ROPE_HALF = 1, AA_ROPE_NONE = 2 } aa_rope_layout;

typedef struct {
  int32_t total_tokens;  /* T >= 2, anchor included; T < 2^30                 */
  int32_t num_q_heads;   /* Hq >= 1                                            */
  int32_t num_kv_heads;  /* Hkv >= 1, Hq % Hkv == 0 (grouped-query attention)  */
  int32_t head_dim;      /* D: 64 or 128                                       */
  double rope_base;      /* theta_p = rope_base^(-2p/D); > 1                   */
  float softmax_scale;   /* <= 0 selects 1/sqrt(D)                             */
  int32_t pos_shift;     /* Delta added to every position (Eq. 3); >= 0       */
  int32_t mask_mode;     /* aa_mask_mode                                       */
  int32_t pos_mode;      /* aa_pos_mode                                        */
  int32_t rope_layout;   /* aa_rope_layout                                     */
  int32_t host_only;     /* 1: build host metadata only (no GPU needed);
                            compute calls on such a plan return
                            AA_ERR_INVALID_ARG                                 */
} aa_config;

typedef struct aa_plan_s* aa_plan_t;

/* Build the plan for one packing [ARCH §3.4 Anchor "Mask construction",
 * §3.4 Index]: per-token document and position IDs, each query row's visible
 * key interval, the live 128x128 tile lists (fully cross-document tiles are
 * dropped; the anchor column is folded in separately) in the order the
 * persistent attention kernels claim them (grouped by document, longest
 * group first: the forward's heads interleaved in each document, the
 * backward's one group per document and head; a forward item is two query
 * tiles of one head, or one query tile of two heads sharing a kv head when
 * Hq/Hkv is even), and the two-level fp32 cos/sin tables of Eq. 6 built in
 * fp64.
 * cu_doclens: host int32[num_docs + 1] (see conventions). Device metadata is
 * uploaded with copies ordered on `stream`. On success *out owns everything;
 * release it with aa_plan_destroy. */
aa_status aa_plan(const aa_config* cfg, const int32_t* cu_doclens_host, int32_t num_docs,
                  aa_stream_t stream, aa_plan_t* out);

/* aa_plan with caller-supplied rotation frequencies: theta (host double[D/2])
 * replaces Eq. 6's theta_p = rope_base^(-2p/D) for every pair p [ARCH §3.4
 * RoPE]; cfg->rope_base is then ignored. This carries the frequency tables of
 * RoPE variants such as NTK-aware scaling or YaRN, which the pages compare
 * with vanilla RoPE for 64K training (architecture page, §3.4 "Long-Context
 * Training Protocol", "Vanilla RoPE vs. NTK vs. YaRN", Table 2) without
 * defining their formulas: the caller computes the table, the library
 * rotates with it (fp64 tables, fp32 rotation, bf16 operands, as for the
 * default). The table is copied. Errors: NULL theta, or an entry that is not
 * finite and >= 0, gives AA_ERR_INVALID_ARG; otherwise as aa_plan. */
aa_status aa_plan_with_theta(const aa_config* cfg, const int32_t* cu_doclens_host, int32_t num_docs,
                             const double* theta, aa_stream_t stream, aa_plan_t* out);

/* Plan for documents given per token, possibly in interleaved chunks
 * [ARCH §3.4 Anchor "Mask construction"]; architecture page, §3.4
 * "AnchorAttention with Interleaved Chunks" (documents split into chunks that
 * are shuffled and recombined with the order inside each document kept).
 * doc_of_token: host int32[T]; token 0 is the anchor and must be 0, every
 * other token names its document with an id >= 1 (any values; chunks of one
 * document share an id, so they see each other; give each chunk its own id
 * to keep chunks apart). A token sees the anchor (ANCHOR mode) and the tokens
 * j <= i of its own document. Positions: RESET counts 1, 2, ... through the
 * document's tokens in order, CONTINUOUS is the token index; pos_shift adds.
 * cfg->mask_mode must be ANCHOR or INTRA_DOC. aa_fwd / aa_bwd /
 * aa_bwd_from_fwd / aa_bwd_static_workspace / aa_rope_apply take and return
 * tensors in the caller's token order (the library's kernels run on the
 * tokens grouped by document: the rotation passes read q and k through the
 * grouping, V is gathered once per forward (aa_bwd_from_fwd reads the
 * forward's copy), the backward's first kernel reads o, dout and lse through
 * it and keeps a grouped dout, and every output is written at its caller
 * position; the workspace sizes include those copies); aa_plan_metadata
 * returns the caller's document ids and
 * positions; aa_plan_stats / aa_plan_work count the grouped layout's tiles.
 * aa_shift_diag refuses segment plans (AA_ERR_UNSUPPORTED). Errors: NULL
 * doc_of_token, doc_of_token[0] != 0, an id < 1 after it, or the aa_plan
 * conditions give AA_ERR_INVALID_ARG. */
aa_status aa_plan_segments(const aa_config* cfg, const int32_t* doc_of_token_host, aa_stream_t stream,
                           aa_plan_t* out);

/* Free a plan (synchronises the device). NULL is accepted. */
aa_status aa_plan_destroy(aa_plan_t plan);

/* Copy the per-token document index (anchor = 0, documents 1..K; all 0 in
 * CAUSAL mode) and position ID (shift included) into caller host buffers of
 * T int32 each. Either pointer may be NULL. */
aa_status aa_plan_metadata(aa_plan_t plan, int32_t* doc_id_host, int32_t* pos_id_host);

/* unmasked_pairs: visible (query, key) pairs of the mask (the T^2/K + T count
 * of [ARCH §3.4 Anchor], "Reduction in attention computations"), anchor pairs
 * included. live_tiles: 128x128 blocks of the mask holding a visible pair.
 * causal_tiles: blocks with any j <= i (what full causal attention visits).
 * Any pointer may be NULL. */
aa_status aa_plan_stats(aa_plan_t plan, int64_t* unmasked_pairs, int64_t* live_tiles,
                        int64_t* causal_tiles);

/* Work the kernels perform: fwd_tiles = (q-tile, k-tile, head) MMA tiles of
 * the forward pass; bwd_tiles = the same count for the backward pass (one
 * tile = one 128x128 block of one query head). Any pointer may be NULL. */
aa_status aa_plan_work(aa_plan_t plan, int64_t* fwd_tiles, int64_t* bwd_tiles);

/* Rotate x [T, num_heads, D] bf16 into y (same shape; y may equal x) with the
 * plan's positions: y = R_pos x (inverse = 0) or R_pos^T x (inverse = 1),
 * fp32 arithmetic, round-to-nearest-even to bf16 [ARCH §3.4 RoPE Eq. 6,
 * ARCH §3.2]. num_heads is independent of the plan's head counts. */
aa_status aa_rope_apply(aa_plan_t plan, const void* x, void* y, int32_t num_heads,
                        int32_t inverse, aa_stream_t stream);

/* Forward [ARCH §3.4 Anchor, §3.4 RoPE]: for every query row i and head h,
 *   O_i = sum_{j visible} softmax_j(scale * (R_i q_i).(R_j k_j)) v_j,
 *   LSE_i = ln sum_{j visible} exp(scale * (R_i q_i).(R_j k_j)).
 * q [T,Hq,D], k/v [T,Hkv,D] bf16 in; o [T,Hq,D] bf16, lse [Hq,T] fp32 out.
 * Query head h reads kv head h / (Hq / Hkv). Q and K are rotated once per
 * call into `workspace` (caller-owned device memory of at least
 * aa_fwd_workspace_bytes(plan) bytes, 256-byte aligned, contents ignored),
 * which the attention kernel then reads; it also holds the kernel's work
 * counter, so forward calls with separate workspaces may overlap. */
aa_status aa_fwd(aa_plan_t plan, const void* q, const void* k, const void* v, void* o,
                 float* lse, void* workspace, size_t workspace_bytes, aa_stream_t stream);

/* Bytes of device scratch aa_fwd needs: the rotated K and Q, T*(Hkv+Hq)*D
 * bf16, which it leaves there for aa_bwd_from_fwd (none with AA_ROPE_NONE),
 * plus 256 bytes for the work counter; segment plans add a grouped copy of
 * v (read again by aa_bwd_from_fwd) and, without RoPE, of q and k. */
size_t aa_fwd_workspace_bytes(aa_plan_t plan);

/* Bytes of device scratch aa_bwd needs (rotated Q and K, fp32 dQ
 * accumulator, per-row D, anchor partial sums; segment plans add their
 * grouped copies). */
size_t aa_bwd_workspace_bytes(aa_plan_t plan);

/* Backward of aa_fwd: given dout = dL/dO, writes dq [T,Hq,D], dk/dv
 * [T,Hkv,D] bf16 = gradients with respect to the UN-ROTATED q, k and v
 * (dq = R^T dq~, dk = R^T dk~). q, k, v, o and lse must be the forward's
 * inputs and outputs. workspace: caller-owned device memory of at least
 * aa_bwd_workspace_bytes(plan) bytes, 256-byte aligned, contents ignored.
 * dK/dV of the anchor sum over every query row (and over the group's query
 * heads). dQ is accumulated with fp32 atomics, so its last bits may vary
 * between runs; every other output is run-to-run deterministic. */
aa_status aa_bwd(aa_plan_t plan, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout, void* dq, void* dk, void* dv,
                 void* workspace, size_t workspace_bytes, aa_stream_t stream);

/* aa_bwd from the forward's rotated operands (no counterpart in the paper:
 * an interface addition of this library) [ARCH §3.4 Anchor, §3.4 RoPE].
 * aa_fwd leaves the rotated Q and K (R_i q_i, R_j k_j, rounded to bf16) in
 * its workspace; a training step that keeps that workspace until the
 * backward pass, instead of q and k, passes it here as fwd_workspace and the
 * backward skips its own rotation of Q and K (two passes over them).
 *  - fwd_workspace: the workspace of an aa_fwd call with this plan and the
 *    q, k whose gradients are wanted, unchanged since that call (the library
 *    cannot check this; it is the caller's contract). Read only.
 *  - v, o, lse, dout, dq, dk, dv: as for aa_bwd; the results are the same
 *    (gradients with respect to the UN-ROTATED q, k and v): dk, dv bit for
 *    bit, dq up to the order of its fp32 atomic additions.
 *  - workspace: at least aa_bwd_from_fwd_workspace_bytes(plan) bytes,
 *    256-byte aligned, contents ignored (smaller than aa_bwd's: no rotated
 *    copies).
 *  - AA_ERR_UNSUPPORTED with AA_ROPE_NONE (aa_fwd rotates nothing; call
 *    aa_bwd); AA_ERR_INVALID_ARG for NULL or misaligned pointers or a short
 *    workspace, with nothing launched. */
aa_status aa_bwd_from_fwd(aa_plan_t plan, const void* fwd_workspace, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          void* workspace, size_t workspace_bytes, aa_stream_t stream);

/* Bytes of device scratch aa_bwd_from_fwd needs. */
size_t aa_bwd_from_fwd_workspace_bytes(aa_plan_t plan);

/* aa_bwd without a caller-provided workspace (no counterpart in the paper:
 * an interface addition of this library).
 * Some callers cannot call cudaMalloc at the point where they run the
 * backward pass: a plugin inside a host framework whose memory planner owns
 * every device allocation, a latency-critical loop where an allocation would
 * stall or synchronise the device, or a deployment that must stay inside a
 * memory budget fixed at start-up. This entry point takes its scratch from a
 * 64 MiB array that the library reserves statically on every GPU that loads
 * it (held until the process exits) and allocates nothing itself.
 *  - Arguments and results are those of aa_bwd minus the workspace pair.
 *  - Plans whose aa_bwd_workspace_bytes() exceeds 64 MiB are rejected with
 *    AA_ERR_INVALID_ARG and a message giving both sizes; nothing is launched.
 *    aa_bwd_workspace_bytes() is the exact test. As a guide, for plans built
 *    from cu_doclens with RoPE at D = 128 a query row needs about 1 KB
 *    (rotated Q and K and the fp32 dQ accumulator) and each query head
 *    64 KB of anchor partials, so T * Hq up to about 60K query rows fit.
 *    Segment plans (aa_plan_segments) also need grouped copies of v and
 *    dout (and, without RoPE, of q and k), so somewhat fewer rows fit.
 *  - The plan's device must be current. The first call on a device looks up
 *    the array's device address (cudaGetSymbolAddress) once and keeps it for
 *    the life of the process; make that first call before any stream capture
 *    on that device. The kept address does not survive a reset of the
 *    device's primary context (cudaDeviceReset): do not call this entry point
 *    after one.
 *  - Every call on a device shares the one array, and the array keeps the
 *    last call's contents; the call overwrites all the scratch it reads, so
 *    nothing needs clearing. Calls whose executions overlap on the GPU (for
 *    instance on two streams) race on the array and give wrong results:
 *    order them on one stream or with events. */
aa_status aa_bwd_static_workspace(aa_plan_t plan, const void* q, const void* k, const void* v,
                                  const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                  void* dv, aa_stream_t stream);

/* Synchronise `stream`, read and clear the plan's device error word.
 * Returns AA_ERR_TIMEOUT if a bounded device wait ran out since the last
 * check, AA_OK otherwise. */
aa_status aa_check_device_error(aa_plan_t plan, aa_stream_t stream);

/* Diagnostics: limit (nanoseconds) of every bounded device wait for this
 * plan; 0 makes each wait give up after its first poll (the kernels then
 * drain their in-flight copies and MMAs and return with the error word set).
 * The default is 2e9 ns. */
aa_status aa_set_wait_limit(aa_plan_t plan, uint64_t nanoseconds);

/* Measurement hook: when both are non-NULL CUDA events (cudaEvent_t),
 * aa_bwd and aa_bwd_from_fwd record `start` immediately before and `stop`
 * immediately after the launch of their main tile kernel, on the call's stream, so that kernel can be
 * timed on its own. NULL, NULL (the default) disables the recording. The
 * events are caller-owned and must outlive the calls that record them. */
aa_status aa_set_bwd_timing_events(aa_plan_t plan, void* start, void* stop);

/* Failure-detection self-test: launches one CTA that waits on a shared-memory
 * barrier nothing ever arrives on, bounded by the plan's wait limit
 * (aa_set_wait_limit). The wait runs out, the kernel records its site code in
 * the plan's error word and returns, leaving the context usable; the next
 * aa_check_device_error() returns AA_ERR_TIMEOUT. This is the same bounded
 * wait every attention kernel uses. */
aa_status aa_selftest_bounded_wait(aa_plan_t plan, aa_stream_t stream);

/* Shift-discrepancy diagnostics. [ARCH §3.4 Diag], [ARCH §3.4 RoPE] (Eq. 3)
 * Two plans that differ only in pos_shift (Δ1 for plan1, Δ2 for plan2) and one
 * un-rotated input q [T, Hq, D], k [T, Hkv, D] (bf16). The library rotates q
 * and k under both shifts with its own RoPE kernel (the bf16 operands its
 * attention uses) and computes, with the plans' mask:
 *   col_absdiff[h][j]         = sum_i |ATTN_ij(Δ1) - ATTN_ij(Δ2)|   (fp32 [Hq, T])
 *   first_logit_absdiff[h][i] = |A_i0(Δ1) - A_i0(Δ2)|              (fp32 [Hq, T])
 *     (0 for rows that cannot see token 0), A = scale * q~_i . k~_j the
 *     pre-softmax logit, ATTN = softmax of A over the visible keys;
 *   result (fp64, 2 + 2*Hq):  result[0] = D (Eq. 4) = sum_h sum_j
 *     col_absdiff[h][j] / n_j with n_j the rows that may attend to key j;
 *     result[1] = D_logit (Eq. 5) = (1/T) sum_h sum_i first_logit_absdiff[h][i];
 *     result[2 + 2h], result[3 + 2h] = head h's two sums.
 * Under exact arithmetic both are zero (Eq. 3); what they measure here is the
 * bf16 rounding of the rotated operands. The logits are recomputed on CUDA
 * cores in fp32 (an evaluation tool, not a training-step kernel); the column
 * sums use atomics, so their last bits can vary run to run.
 * workspace: aa_shift_diag_workspace_bytes(plan1) bytes (rotated Q and K under
 * both shifts; 0 without RoPE), 16-byte aligned device memory. Errors: plans
 * that differ in anything but pos_shift, a host-only plan, NULL or unaligned
 * pointers, or a short workspace give AA_ERR_INVALID_ARG before any launch. */
size_t aa_shift_diag_workspace_bytes(aa_plan_t plan);
aa_status aa_shift_diag(aa_plan_t plan1, aa_plan_t plan2, const void* q, const void* k, float* col_absdiff,
                        float* first_logit_absdiff, double* result, void* workspace, size_t workspace_bytes,
                        aa_stream_t stream);

/* Sharding of one packing across ranks [ARCH §3.4 Anchor] ("Mask
 * construction": documents see nothing of one another; every row sees the
 * anchor), architecture page §3.4 "AnchorContext: Implementation
 * Infrastructure" (the pages shard attention over 8 GPUs). Host only: no
 * plan, no device.
 * A piece is document `doc` (1-based, as in cu_doclens) restricted to kv
 * heads [kv_head_begin, kv_head_end) and their query heads (query head h
 * belongs to kv head h / group); `cost` = its visible pairs, (N(N+1)/2 + N)
 * per query head. Pieces go longest first to the least-loaded shard; a
 * document whose all-head cost exceeds total / num_shards is first cut into
 * ceil(cost / (total / num_shards)) kv-head ranges (at most num_kv_heads).
 * Every (document, kv head) lies in exactly one piece, so each rank runs its
 * pieces as ordinary packings (one per distinct head range, each with its
 * own copy of the anchor token) and the only exchanges are the anchor's k_0 /
 * v_0 (broadcast before the forward) and the sum of the ranks' dk_0 / dv_0
 * (all-reduce after the backward).
 *  - cu_doclens: host int32[num_docs + 1], as for aa_plan (cu[0] == 1).
 *  - group = Hq / Hkv; num_shards >= 1.
 *  - pieces: caller array of max_pieces entries, filled sorted by (shard,
 *    kv_head_begin, doc); *num_pieces receives the count. If max_pieces is
 *    too small, *num_pieces receives the count needed and AA_ERR_INVALID_ARG
 *    is returned (call with pieces = NULL, max_pieces = 0 to size the array).
 *  - shard_cost: optional int64[num_shards], each shard's summed cost. */
typedef struct {
  int32_t shard, doc, kv_head_begin, kv_head_end;
  int64_t cost;
} aa_shard_piece;
aa_status aa_shard_plan(const int32_t* cu_doclens_host, int32_t num_docs, int32_t num_kv_heads, int32_t group,
                        int32_t num_shards, aa_shard_piece* pieces, int32_t max_pieces, int32_t* num_pieces,
                        int64_t* shard_cost);

const char* aa_status_string(aa_status status);
const char* aa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ANCHORATTN_H */
