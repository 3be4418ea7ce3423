/*
 * tpk.h -- C ABI of the prefix-tree-packed DFS attention library (GB300, sm_103a).
 *
 * The library computes attention over training rows packed as a prefix tree:
 * sequences that share a token prefix are laid out once, depth first, in
 * fixed-capacity rows; every token attends only to itself and its
 * root-to-leaf ancestors; position ids are tree depths; a token_index maps
 * every raw token back to its forwarded position.  The pages that define the
 * method:
 *   [ART]  "Prefix Tree Packing in ART" -- sections "The tree" (recursive
 *          longest-run walk, minimum shared-segment length, duplicated join
 *          token), "One tree, not one per group", "Bin packing, with a twist"
 *          (best-fit decreasing over marginal cost), "Token-mixing layers"
 *          (tree mask = full ancestor blocks + causal own block; [enter, exit]
 *          interval ancestor test), "Metadata space first".
 *   [DAG]  "DAG packing" -- sections "The walk" (depth-first layout, last
 *          common node copied per child), "The mask", "Positions" (depth).
 *   [TRL]  "TRL Tree Packing for AsyncGRPO" -- section "How tree packing
 *          works" (planner -> collator -> attention; token_index).
 *
 * Conventions for every call
 *  - Return value: TPK_OK (0) or a negative TPK_E_* code; tpk_status_string()
 *    names it.  No call aborts the process.
 *  - Memory: the library never allocates device memory.  The caller owns
 *    every device buffer (PyTorch in the bundled binding) and the stream.
 *    Plan handles live in host memory owned by the library until
 *    tpk_plan_destroy().
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  GPU calls only enqueue work; they never synchronise.
 *  - Layouts (row-major, contiguous):
 *      Q, O      [F, Hq, d]  bf16, forwarded order (rows concatenated)
 *      K, V      [F, Hkv, d] bf16
 *      LSE       [Hq, F]     fp32, natural log
 *      raw-order outputs: [R, Hq, d] bf16 and [Hq, R] fp32, raw order = the
 *      concatenation of the input sequences by seq_offsets.
 *    Grouped-query attention: query head h reads key/value head h / (Hq/Hkv).
 *  - Device errors: attention kernels bound every wait; a wait that gives up
 *    writes TPK_E_TIMEOUT to *dev_err (device int32, caller-initialised to 0)
 *    and the kernel exits cleanly.  Read it after synchronising.
 *  - There is no CPU fallback: GPU entry points return TPK_E_CUDA or
 *    TPK_E_UNSUPPORTED when no sm_103 device is usable.
 */
#ifndef TPK_H_
#define TPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define TPK_OK               0
#define TPK_E_ARG           -1  /* bad argument (NULL pointer, size, offsets) */
#define TPK_E_SEQ_TOO_LONG  -2  /* a sequence is longer than row_capacity */
#define TPK_E_OVERFLOW      -3  /* F, R or a table size does not fit int32 */
#define TPK_E_UNSUPPORTED   -4  /* head_dim not in {64,128}, Hq % Hkv != 0, no sm_103 device */
#define TPK_E_CUDA          -5  /* a CUDA runtime/driver call failed */
#define TPK_E_TIMEOUT       -6  /* a device wait gave up (read from dev_err) */
#define TPK_E_WORKSPACE     -7  /* workspace missing or smaller than required */
#define TPK_E_SCRATCH_LIMIT -8  /* problem too large for tpk_tree_attn_bwd_noalloc's static scratch */
#define TPK_E_HOST          -9  /* host-side failure in the planner: out of host memory or
                                   another C++ exception, caught before it reaches the caller */

/* ---- placement rules ---------------------------------------------------- */
#define TPK_PLACE_BFD       0   /* [ART] "Bin packing, with a twist": best-fit decreasing
                                   over marginal cost (the default) */
#define TPK_PLACE_NEXT_FIT  1   /* [ART] "One tree, not one per group": fill rows in
                                   order, open a new row when the next leaf does not fit */
#define TPK_PLACE_GROUPS    2   /* no counterpart on the pages: one row per placement
                                   group, rows in increasing group id (a rank that owns
                                   rows of a larger batch, see tpk_plan_shard_rows, plans
                                   its sequences with their global row as the group and
                                   gets those rows back); a group that does not fit in
                                   one row gives TPK_E_SEQ_TOO_LONG */

typedef struct tpk_plan tpk_plan;   /* opaque, host memory */

typedef struct {
    int64_t row_capacity;  /* forwarded tokens per row ([ART] intro: row length set by
                              memory; [TRL] token_budget counts forwarded tokens) */
    int32_t min_shared;    /* minimum shared-segment length ([ART] "The tree": shorter
                              shared runs are copied into each branch); <=1 disables */
    int32_t placement;     /* TPK_PLACE_BFD, TPK_PLACE_NEXT_FIT or TPK_PLACE_GROUPS */
} tpk_plan_opts;

typedef struct {
    int64_t n_seqs;        /* input sequences */
    int64_t n_rows;        /* packed rows */
    int64_t n_fwd;         /* F: forwarded positions over all rows */
    int64_t n_raw;         /* R: raw tokens */
    int64_t n_segments;    /* segments of the global prefix tree */
    int64_t n_leaves;      /* distinct sequences */
    int64_t n_qtiles;      /* 128-query tiles (forward work list) */
    int64_t n_kblocks;     /* key blocks over all query tiles */
    int64_t n_ktiles;      /* 128-key tiles (backward work list) */
    int64_t n_qblocks;     /* query blocks over all key tiles */
    int64_t useful_pairs;  /* sum over forwarded f of depth[f]+1: visible (query, key) pairs */
    int64_t visited_pairs; /* query rows x key columns the forward kernel visits */
    int64_t max_depth;
    double packing_ratio;  /* R / F ([TRL] "How tree packing works") */
    double row_fill_frac;  /* F / (n_rows * row_capacity) */
    double fork_frac;      /* segments with >= 2 children / segments */
    int64_t n_seg_instances; /* segment instances (a segment placed in one row), see tpk_plan_segments */
    int64_t n_seg_levels;    /* tree levels of the segment instances */
} tpk_plan_info;

/* ---- planner (host only, no GPU needed) --------------------------------- */

/* Build the packing plan ([ART] "The tree", "Bin packing, with a twist";
 * [DAG] "The walk", "Positions"; [TRL] "How tree packing works").
 *   tokens      [R] int32 token ids >= 0, sequences concatenated
 *   seq_offsets [n_seqs+1] int64, seq_offsets[0] = 0, strictly increasing
 *               (every sequence has >= 1 token), seq_offsets[n_seqs] = R
 *   trained     [R] uint8 or NULL (= all 1): 1 if the position's next-token
 *               prediction carries a loss.  A position is shared only when
 *               the token prefix, the flags and -- for a trained position --
 *               its target agree, so the last common token before a fork is
 *               kept once per branch ([ART] "The tree", off-by-one note).
 *   group_ids   [n_seqs] int32 or NULL: placement groups (best-fit decreasing
 *               orders groups by their most expensive leaf).  NULL = the tree
 *               family (root segment) of each sequence.
 *   opts        see tpk_plan_opts (NULL = capacity 65536, min_shared 64, BFD)
 *   out         receives the new plan; free with tpk_plan_destroy.
 * The planner uses up to 16 host threads (the environment variable
 * TPK_PLANNER_THREADS sets another limit, >= 1); its result does not
 * depend on the number.
 * Errors: TPK_E_ARG (bad offsets / negative token / NULL), TPK_E_SEQ_TOO_LONG,
 *         TPK_E_OVERFLOW (F or R >= 2^31), TPK_E_HOST (host memory exhausted or
 *         another exception inside the planner; no exception crosses the ABI).
 *         If fewer worker threads can be created than asked for, the planner
 *         runs on the ones it has (same result).  Inputs are copied; the caller
 *         keeps ownership of its buffers. */
int tpk_plan_build(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
                   const uint8_t* trained, const int32_t* group_ids,
                   const tpk_plan_opts* opts, tpk_plan** out);

int tpk_plan_info_get(const tpk_plan* plan, tpk_plan_info* out);

/* Copy the layout into caller-allocated host buffers (any pointer may be NULL):
 *   row_offsets [n_rows+1] forwarded offset of each row
 *   row_loads   [n_rows]   forwarded tokens of each row
 *   row_of_seq  [n_seqs]
 *   fwd_token   [F]  token id at each forwarded position
 *   fwd_src     [F]  lowest raw index that maps to the position (its owner)
 *   parent      [F]  forwarded index of the position one level up, -1 at a root
 *   depth       [F]  tree depth = position id ([DAG] "Positions")
 *   token_index [R]  forwarded index of every raw token ([TRL])
 *   subtree_end [F]  one past the last position of the subtree: key j is visible
 *                    to query i iff j <= i < subtree_end[j] ([ART] "Token-mixing
 *                    layers", [enter, exit] interval test) */
int tpk_plan_export(const tpk_plan* plan, int64_t* row_offsets, int64_t* row_loads,
                    int32_t* row_of_seq, int32_t* fwd_token, int32_t* fwd_src,
                    int32_t* parent, int32_t* depth, int32_t* token_index,
                    int32_t* subtree_end);

/* Kernel work lists (int32, host copies; any pointer may be NULL).
 * Forward: query tile t covers forwarded [qt_q0[t], qt_q0[t]+qt_nq[t]) inside one
 * row; its key blocks are kb[2*b], kb[2*b+1] for b in [qt_kb_begin[t],
 * qt_kb_begin[t+1]): kb[2b] = first key, kb[2b+1] = count | (full << 16), where
 * full = the block has 128 keys and every one is visible to every query of the
 * tile (the kernel then skips the mask).  The
 * key set of a tile is the ancestors of its first query plus the tile itself
 * (a contiguous ancestor chain of segment intervals, [ART] "Token-mixing layers").
 * Backward: key tile u covers [kt_k0[u], +kt_nk[u]); its query blocks qb[2c],
 * qb[2c+1] for c in [kt_qb_begin[u], kt_qb_begin[u+1]) cover [k0, max subtree_end).
 * qt_order / kt_order: launch order of the tiles.  Tiles are cut into runs of
 * 128 consecutive tiles (depth-first order); runs come by decreasing total
 * work, and inside a run tiles come by decreasing work.  Neighbouring tiles
 * share ancestor (query tiles) or descendant (key tiles) blocks, so CTAs that
 * run together reuse them from L2. */
int tpk_plan_worklists(const tpk_plan* plan, int32_t* qt_q0, int32_t* qt_nq,
                       int32_t* qt_kb_begin, int32_t* kb, int32_t* qt_order,
                       int32_t* kt_k0, int32_t* kt_nk, int32_t* kt_qb_begin,
                       int32_t* qb, int32_t* kt_order);

/* Raw tokens of each forwarded position: token_index read the other way, as
 * a CSR (int32 host copies; either pointer may be NULL).
 * fwd_raw[fwd_raw_begin[f] .. fwd_raw_begin[f+1]) lists, ascending, the raw
 * tokens that map to forwarded position f; the first is fwd_src[f], its owner.
 * fwd_raw_begin has F+1 entries, fwd_raw R.  The device image holds the same
 * arrays (TPK_FIELD_FWD_RAW_BEGIN, TPK_FIELD_FWD_RAW) for
 * tpk_gather_to_forwarded and tpk_sum_to_forwarded. */
int tpk_plan_raw_of_forwarded(const tpk_plan* plan, int32_t* fwd_raw_begin, int32_t* fwd_raw);

/* Segment instances by tree level ([ART] "Token-mixing layers", GDN: a
 * recurrent layer threads its state through the tree one depth at a time --
 * every segment of a depth, across all rows, in one pass -- and a child
 * starts from its parent's final state, a root from zero).  An instance is a
 * segment placed in one row: a chain of forwarded positions [seg_start,
 * seg_start + seg_len).  Instances are ordered by level (the number of
 * ancestor instances), then by placement; level l is [level_begin[l],
 * level_begin[l+1]) (n_seg_levels + 1 entries); seg_parent is the parent's
 * index in this order, -1 at a root.  Host int32 copies, any pointer may be
 * NULL; sizes from tpk_plan_info (n_seg_instances, n_seg_levels).  The
 * device image holds seg_start, seg_len, seg_parent and seg_off, the number
 * of positions of the instances before it on its level (TPK_FIELD_SEG_*).
 * Within a level instances are in ascending seg_start, so the children of an
 * instance are one contiguous run of the next level. */
int tpk_plan_segments(const tpk_plan* plan, int32_t* level_begin, int32_t* seg_start, int32_t* seg_len,
                      int32_t* seg_parent);

/* Rows across ranks (no counterpart on the pages, which run one GPU per
 * row batch): the mask never crosses a row ("Prefix Tree Packing in ART",
 * section "Token-mixing layers": a token sees only its own root-to-leaf
 * path), so rows are independent units of work and data-parallel ranks can
 * take whole rows with nothing exchanged.  A row's work is its useful
 * (query, key) pairs, the sum of depth + 1 over its forwarded positions.
 * Rows are assigned longest first, each to the rank with the least work so
 * far (ties: lower row index first, then the lower rank), which keeps every
 * rank's total within one row's work of the lightest rank's.
 *   rank_of_row: host int32 [n_rows], written (rank 0 .. world-1 per row);
 *   rank_pairs:  host int64 [world], each rank's total pairs (may be NULL).
 * A rank runs the sequences whose row it owns (row_of_seq of
 * tpk_plan_export), planned as a batch of their own with their global row
 * as the group and TPK_PLACE_GROUPS, which gives back exactly those rows.
 * Returns TPK_E_ARG for
 * a NULL plan or rank_of_row, or world <= 0. */
int tpk_plan_shard_rows(const tpk_plan* plan, int32_t world, int32_t* rank_of_row, int64_t* rank_pairs);

/* Device image of the plan.  The caller allocates tpk_plan_device_bytes()
 * bytes of device memory (256-byte aligned) and uploads the image with
 * tpk_plan_upload (async on `stream`; the plan keeps the host image alive until
 * destroyed, so keep the plan until the copy has completed).  The first upload
 * copies the image once into page-locked host memory owned by the plan, so
 * every upload is an asynchronous DMA.  tpk_plan_destroy hands that buffer
 * to the next plan's upload instead of freeing it (the library keeps at most
 * two such buffers per process: allocating and freeing page-locked memory
 * costs more than the copy).  If page-locked memory cannot be had, the
 * upload copies from pageable memory (same bytes, not asynchronous).
 * tpk_plan_field_offset gives the byte offset of a field inside
 * the image so callers can pass e.g. depth or token_index to the kernels. */
#define TPK_FIELD_DEPTH        0   /* int32 [F] */
#define TPK_FIELD_TOKEN_INDEX  1   /* int32 [R] */
#define TPK_FIELD_SUBTREE_END  2   /* int32 [F] */
#define TPK_FIELD_PARENT       3   /* int32 [F] */
#define TPK_FIELD_FWD_RAW_BEGIN 4  /* int32 [F+1] */
#define TPK_FIELD_FWD_RAW      5   /* int32 [R] */
#define TPK_FIELD_SEG_START    6   /* int32 [n_seg_instances], level order (tpk_plan_segments) */
#define TPK_FIELD_SEG_LEN      7   /* int32 [n_seg_instances] */
#define TPK_FIELD_SEG_PARENT   8   /* int32 [n_seg_instances] */
#define TPK_FIELD_SEG_OFF      9   /* int32 [n_seg_instances]: positions of the instances before it on its level */
size_t tpk_plan_device_bytes(const tpk_plan* plan);
int tpk_plan_field_offset(const tpk_plan* plan, int32_t field, size_t* offset);
int tpk_plan_upload(const tpk_plan* plan, void* dev_image, void* stream);

/* Frees the plan.  The library keeps the host arrays of the last destroyed
 * plan (at most one plan's worth) and builds the next tpk_plan_build into
 * them, so a loop that plans one batch per step writes into memory that is
 * already mapped.  NULL is ignored. */
void tpk_plan_destroy(tpk_plan* plan);

/* ---- GPU kernels (sm_103a) ---------------------------------------------- */

/* RoPE at depth positions ([DAG] "Positions": position id = graph depth, so
 * every parent->child edge has relative distance 1).  Rotates q_in [F,Hq,d]
 * into q_out and k_in [F,Hkv,d] into k_out (bf16; out == in is allowed and
 * rotates in place; a NULL pair skips that tensor).  Pair i < d/2 is
 * (x_i, x_{i+d/2}) rotated by angle depth[f] * base^(-2i/d) (by minus that
 * angle when `inverse` != 0, which maps gradients w.r.t. rotated inputs back
 * to the un-rotated ones).  Math in fp32 with the angle reduced to a fraction
 * of a turn in fp64; output rounded to nearest even.  depth: device int32
 * [F].  d in {64, 128}.  Input and output must not partially overlap. */
int tpk_rope_by_depth(const void* q_in, const void* k_in, void* q_out, void* k_out,
                      const int32_t* depth, int64_t F, int32_t Hq, int32_t Hkv, int32_t d,
                      double base, int32_t inverse, void* stream);

/* Options of the attention calls (tpk_tree_attn_fwd_ex, tpk_tree_attn_bwd_ex).
 * No counterpart on the pages: they choose the arithmetic, not the result.
 *   precision  TPK_PREC_FAST: the probabilities P (forward and backward) and
 *              the score gradients dS (backward) enter their tensor-core
 *              products as bf16, as in any bf16 flash-attention kernel.  The
 *              backward's error is then about 1.3% of max(1, |gradient|) at
 *              worst on unit-variance inputs, against 0.4% for the bf16
 *              rounding of the gradient itself.
 *              TPK_PREC_PRECISE: each of P and dS is split into a bf16 high
 *              part and the bf16 rounding of the remainder, and both parts
 *              are multiplied (two products where the fast mode has one), so
 *              they carry about 16 significant bits.  The forward also returns
 *              O's rounding residual (o_lo), and the backward's row terms
 *              D = dO . O use it, so D is taken from O before its bf16 rounding.
 *              dQ, dK and dV then differ from the exact gradients by about the
 *              bf16 rounding of the outputs alone.  Costs one more product for
 *              each of PV, dV, dK and dQ.
 *   rope_base  backward only: > 1 returns dq and dk with respect to the
 *              un-rotated q and k -- the inverse of tpk_rope_by_depth at depth
 *              ("DAG packing", section "Positions") is applied to the fp32
 *              gradients in the kernels' epilogues, before their one bf16
 *              rounding -- so no inverse RoPE pass is needed; the plan's depths
 *              must be below 2^24 (TPK_E_UNSUPPORTED otherwise).  0 = with
 *              respect to the rotated inputs (no rotation).
 *   o_lo       [F, Hq, d] bf16, 16-byte aligned.  Forward, precise: output,
 *              bf16(O - bf16(O)) of the fp32 output (NULL: not written).
 *              Backward, precise: input, D = dO . (o + o_lo) (NULL: D = dO . o).
 *              Ignored in the fast mode.
 * A NULL options pointer means fast, no rotation, no o_lo. */
#define TPK_PREC_FAST     0
#define TPK_PREC_PRECISE  1
typedef struct {
    int32_t precision;   /* TPK_PREC_FAST or TPK_PREC_PRECISE */
    int32_t reserved;    /* 0 */
    double rope_base;    /* backward: 0, or > 1 for gradients w.r.t. the un-rotated q, k */
    void* o_lo;          /* see above */
} tpk_attn_opts;

/* Workspace bytes for the attention calls (0 for the forward). */
size_t tpk_attn_workspace_bytes(const tpk_plan* plan, int32_t Hq, int32_t Hkv,
                                int32_t d, int32_t backward);

/* Tree attention forward ([ART] "Token-mixing layers"; [DAG] "The mask"):
 * O[f,h] = sum over keys j visible to f of softmax_j(scale * q_f . k_j) v_j,
 * visible = f itself and its ancestors (j <= f < subtree_end[j]);
 * LSE[h,f] = ln sum_j exp(scale * q_f . k_j).  q, k are the RoPE-rotated
 * inputs.  Only key blocks on the query tile's ancestor chain are visited,
 * so work scales with forwarded tokens, not raw ones.
 *   plan/dev_image  the plan and its uploaded image
 *   q [F,Hq,d], k/v [F,Hkv,d], o [F,Hq,d] bf16 (device, 16-byte aligned)
 *   lse [Hq,F] fp32 (device)
 *   d in {64,128}; Hq % Hkv == 0; scale > 0 (usually 1/sqrt(d))
 *   workspace/ws_bytes: may be NULL/0 (none needed)
 *   dev_err: device int32 set to TPK_E_TIMEOUT if a wait gave up (may be NULL) */
int tpk_tree_attn_fwd(const tpk_plan* plan, const void* dev_image,
                      const void* q, const void* k, const void* v,
                      void* o, float* lse, int32_t Hq, int32_t Hkv, int32_t d,
                      float scale, void* workspace, size_t ws_bytes,
                      int32_t* dev_err, void* stream);

/* tpk_tree_attn_fwd with options (precision, O's rounding residual; see
 * tpk_attn_opts).  rope_base must be 0 (the forward takes rotated q, k).
 * Same arguments and errors as tpk_tree_attn_fwd otherwise. */
int tpk_tree_attn_fwd_ex(const tpk_plan* plan, const void* dev_image,
                         const void* q, const void* k, const void* v,
                         void* o, float* lse, int32_t Hq, int32_t Hkv, int32_t d,
                         float scale, const tpk_attn_opts* opts,
                         int32_t* dev_err, void* stream);

/* Tree attention backward: gradients of sum_{f,h} <dout[f,h], O[f,h]> w.r.t.
 * the rotated q and k and w.r.t. v (apply tpk_rope_by_depth(inverse=1) to dq
 * and dk for the un-rotated inputs).  o and lse are the forward's outputs.
 * dk, dv are summed over the query heads of each key/value head.  The result
 * is deterministic (no atomics): dK/dV come from a key-major pass over each
 * key tile's descendants, dQ from a query-major pass over the forward's
 * ancestor blocks.
 *   workspace: >= tpk_attn_workspace_bytes(plan, Hq, Hkv, d, 1) bytes, 256-byte
 *   aligned (fp32 row terms D = dO.O); contents need not be cleared. */
int tpk_tree_attn_bwd(const tpk_plan* plan, const void* dev_image,
                      const void* q, const void* k, const void* v,
                      const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv,
                      int32_t d, float scale, void* workspace, size_t ws_bytes,
                      int32_t* dev_err, void* stream);

/* One phase of tpk_tree_attn_bwd (same arguments), for callers that time or
 * schedule the phases separately.  Phases must run in order 0, then 1 and 2
 * (1 and 2 are independent of each other):
 *   TPK_BWD_PREP  D[h,f] = dout[f,h] . o[f,h] into the workspace
 *   TPK_BWD_DKDV  key-major pass: dk, dv
 *   TPK_BWD_DQ    query-major pass: dq
 * Arguments a phase does not read may be NULL. */
#define TPK_BWD_ALL  -1   /* tpk_tree_attn_bwd_ex only: phases 0, 1, 2 in order */
#define TPK_BWD_PREP 0
#define TPK_BWD_DKDV 1
#define TPK_BWD_DQ   2
int tpk_tree_attn_bwd_phase(int32_t phase, const tpk_plan* plan, const void* dev_image,
                            const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout,
                            void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv,
                            int32_t d, float scale, void* workspace, size_t ws_bytes,
                            int32_t* dev_err, void* stream);

/* tpk_tree_attn_bwd / tpk_tree_attn_bwd_phase with options (see
 * tpk_attn_opts): precision, the forward's rounding residual of O, and the
 * inverse RoPE fused into the epilogues.  phase = TPK_BWD_ALL runs the three
 * phases in order; one phase runs that phase alone (same rules as
 * tpk_tree_attn_bwd_phase).  Deterministic in both precisions.  Errors as
 * tpk_tree_attn_bwd; TPK_E_ARG also for an unknown precision or a rope_base
 * that is neither 0 nor > 1. */
int tpk_tree_attn_bwd_ex(int32_t phase, const tpk_plan* plan, const void* dev_image,
                         const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv,
                         int32_t d, float scale, const tpk_attn_opts* opts,
                         void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/* Backward for callers that cannot allocate device memory at call time.
 * The pages have no counterpart: this is a deployment variant of
 * tpk_tree_attn_bwd.  Some hosts own all device memory and give plugins
 * none when they run; some callers must not call cudaMalloc/cudaFree because
 * those can synchronise the device; some C runtimes have no device allocator.
 * This entry point takes the same inputs and outputs as tpk_tree_attn_bwd but
 * no workspace: its scratch (fp32 D = dO.O, Hq * F * 4 bytes) is a fixed
 * 32 MiB array inside the library, which every GPU that loads the library
 * keeps until the process exits.  Problems with Hq * F > 8,388,608 return
 * TPK_E_SCRATCH_LIMIT (use tpk_tree_attn_bwd with a workspace instead).
 * The first call in each CUDA context -- per device, for the runtime's
 * primary contexts -- looks up the array's device address in that context;
 * make that first call before any stream capture.  The address is cached by
 * the context's unique id, so a context created after cudaDeviceReset, or
 * another context the caller makes current, gets its own lookup.
 * Every call on a device shares the one array, so calls that overlap on the
 * GPU (different streams without ordering) race; calls on one stream are
 * ordered and safe.  Nothing needs clearing: each call overwrites the part it
 * reads.  Results are identical to tpk_tree_attn_bwd's. */
int tpk_tree_attn_bwd_noalloc(const tpk_plan* plan, const void* dev_image,
                              const void* q, const void* k, const void* v,
                              const void* o, const float* lse, const void* dout,
                              void* dq, void* dk, void* dv, int32_t Hq, int32_t Hkv,
                              int32_t d, float scale, int32_t* dev_err, void* stream);

/* Scatter forwarded outputs back to raw-token order ([TRL] "How tree packing
 * works": token_index maps each raw token to its forwarded position):
 *   dst[r] = src[token_index[r]]            src [F,H,d] -> dst [R,H,d] bf16
 *   lse_dst[h,r] = lse_src[h,token_index[r]]  [H,F] -> [H,R] fp32
 * lse_src/lse_dst may both be NULL; src/dst may both be NULL. */
int tpk_scatter_token_index(const int32_t* token_index, int64_t R, int64_t F,
                            const void* src, void* dst, const float* lse_src,
                            float* lse_dst, int32_t H, int32_t d, void* stream);

/* Materialisation of per-token data into the packed layout ([ART] "Metadata
 * space first": once the plan is fixed, one pass slices token ids, logprobs,
 * advantages and other per-token payloads into the packed tensors).  Every
 * forwarded position takes the row of its owner, the lowest raw token that
 * maps to it (fwd_raw[fwd_raw_begin[f]], = fwd_src[f]):
 *   dst[f, :] = src[fwd_src[f], :]      src [R, row_bytes] -> dst [F, row_bytes]
 * Rows are opaque bytes (any element type); row_bytes >= 1.  Merged raw
 * tokens carry the same token and target, so for payloads that are functions
 * of (prefix, target) -- token ids, reference logprobs -- every raw token of
 * a position holds the owner's value.  fwd_raw_begin / fwd_raw: device
 * pointers into the plan image (TPK_FIELD_FWD_RAW_BEGIN / _FWD_RAW).
 * src/dst are device buffers that must not overlap.  Returns TPK_E_ARG on a
 * NULL pointer or negative size, TPK_E_CUDA on a launch error. */
int tpk_gather_to_forwarded(const int32_t* fwd_raw_begin, const int32_t* fwd_raw, int64_t F, int64_t R,
                            const void* src, void* dst, int64_t row_bytes, void* stream);

/* Adjoint of tpk_scatter_token_index: per-raw-token quantities summed into
 * the forwarded position every raw token maps to (no counterpart on the pages
 * beyond [TRL]'s token_index; it is the transpose of that gather, which is how
 * raw-order output gradients -- and per-token loss weights such as
 * advantages -- reach the packed layout):
 *   dst[f]        = sum over r with token_index[r] = f of src[r]      [R,H,d] -> [F,H,d] bf16
 *   lse_dst[h, f] = sum over the same r of lse_src[h, r]               [H,R]  -> [H,F]  fp32
 * Sums run in fp32 over the raw tokens in ascending order (deterministic),
 * then round to bf16 (RNE) for dst.  A per-token fp32 weight [R] is the lse
 * pair with H = 1.  src/dst may both be NULL; lse_src/lse_dst may both be
 * NULL.  H*d*2 must be a multiple of 16 and src/dst 16-byte aligned
 * (TPK_E_ARG otherwise). */
int tpk_sum_to_forwarded(const int32_t* fwd_raw_begin, const int32_t* fwd_raw, int64_t F, int64_t R,
                         const void* src, void* dst, const float* lse_src, float* lse_dst,
                         int32_t H, int32_t d, void* stream);

/* ---- GDN (Gated DeltaNet) token mixing over the tree ---------------------
 * [ART] "Token-mixing layers": GDN is recurrent -- a running state threaded
 * token by token along each root-to-leaf path, forked once per branch point,
 * reset at every tree root -- and runs as a short causal convolution followed
 * by the gated delta rule.  The pages name the layer without defining it; the
 * library computes the published Gated DeltaNet layer, below. */

/* Causal depthwise convolution + SiLU along every position's own path:
 *   y[f, c] = silu( sum_{j<W} w[c, j] * x[a_{W-1-j}(f), c] ),
 * a_0(f) = f, a_{t+1}(f) = parent(a_t(f)); taps above a root read 0.  One
 * launch covers the whole packed batch (each position gathers its window
 * through the plan's parent array).
 *   x, y  [F, C] bf16 device, 16-byte aligned rows; C % 8 == 0
 *   w     [C, W] fp32 device, 16-byte aligned; 1 <= W <= 8
 * Errors: TPK_E_ARG on a NULL pointer, a bad C / W or misalignment. */
int tpk_gdn_conv(const tpk_plan* plan, const void* dev_image, const void* x, const float* w, void* y,
                 int32_t C, int32_t W, void* stream);

/* Workspace of tpk_gdn_delta_rule: one fp32 dv x dk state per segment
 * instance and head (n_seg_instances * H * dk * dv * 4 bytes, rounded up to
 * 256). */
size_t tpk_gdn_workspace_bytes(const tpk_plan* plan, int32_t H, int32_t dk, int32_t dv);

/* The gated delta rule along every root-to-leaf path, per head h:
 *   k~ = k / |k|,  q~ = q / |q|   (L2 over dk; k and q must be nonzero)
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k~_t k~_t^T) + beta_t v_t k~_t^T,  S = 0 at a root
 *   o_t = S_t (scale q~_t)
 * S is dv x dk, kept in fp32.  The segment instances of the plan run level by
 * level (tpk_plan_segments), one launch per level and one CTA per (instance,
 * head): a chain starts from its parent's final state, stored in the
 * workspace, so the state is forked at every branch point.
 *   q, k   [F, H, dk] bf16 with row stride ld_qk elements (may be column
 *          slices of one [F, ld] tensor, e.g. the convolution's output)
 *   v      [F, H, dv] bf16 with row stride ld_v
 *   g, beta [F, H] fp32: log decay (<= 0) and write strength
 *   o      [F, H, dv] bf16 (contiguous)
 *   (dk, dv) in {(64, 64), (128, 128)}; scale > 0 (usually 1/sqrt(dk))
 *   workspace: >= tpk_gdn_workspace_bytes bytes, 256-byte aligned; need not be
 *   cleared.  It holds the final states of the chains that have children
 *   afterwards: keep it unchanged for tpk_gdn_delta_rule_bwd (its `state`).
 * Pointers and strides must give 16-byte aligned rows (TPK_E_ARG). */
int tpk_gdn_delta_rule(const tpk_plan* plan, const void* dev_image, const void* q, const void* k, const void* v,
                       int64_t ld_qk, int64_t ld_v, const float* g, const float* beta, void* o, int32_t H,
                       int32_t dk, int32_t dv, float scale, void* workspace, size_t ws_bytes, void* stream);

/* Gradients of tpk_gdn_conv ("Prefix Tree Packing in ART", section
 * "Token-mixing layers": the layer is differentiated through the packed
 * tree, a position's input feeding the windows of its descendants on every
 * branch below it).  For the output gradient dy [F, C] bf16:
 *   dx[f, c] = sum over f' = f and the descendants of f within W-1 steps of
 *              w[c, W-1-t] dy[f', c] silu'(a[f', c])    (t: steps from f to f')
 *   dw[c, j] = sum_f dy[f, c] silu'(a[f, c]) x[a_{W-1-j}(f), c]
 * with a the convolution's pre-activation (recomputed from x and w).
 *   x, dy, dx [F, C] bf16; w [C, W] fp32 (16-byte aligned); dw [C, W] fp32,
 *   overwritten (summed in a fixed order: deterministic).
 *   workspace: >= tpk_gdn_conv_bwd_workspace_bytes bytes (per-stream partial
 *   sums of dw), 256-byte aligned, need not be cleared.
 * Same argument rules as tpk_gdn_conv; TPK_E_WORKSPACE for a short or
 * misaligned workspace. */
size_t tpk_gdn_conv_bwd_workspace_bytes(const tpk_plan* plan, int32_t C, int32_t W);
int tpk_gdn_conv_bwd(const tpk_plan* plan, const void* dev_image, const void* x, const float* w, const void* dy,
                     void* dx, float* dw, int32_t C, int32_t W, void* workspace, size_t ws_bytes, void* stream);

/* Gradients of tpk_gdn_delta_rule for the output gradient dout [F, H, dv]
 * bf16 (contiguous): dq, dk w.r.t. the un-normalised q, k ([F, H, dk] bf16,
 * row stride ld_dqk), dv ([F, H, dv] bf16, row stride ld_dv), dg, dbeta
 * ([F, H] fp32).  "Prefix Tree Packing in ART", section "Token-mixing
 * layers": a child's initial state is its parent's final state, so the
 * gradient of that state is the sum over the children; here each instance,
 * deepest level first, hands the gradient of its initial state to its
 * parent, which adds those of all its children (ascending order: the result
 * is deterministic) before running its own chain backwards.  The state of
 * each chain is recomputed from its initial state; dk = dv in {64, 128}.
 *   q, k, v, ld_qk, ld_v, g, beta, H, dk, dv, scale: as given to the forward.
 *   state: the workspace the forward filled (its saved final states; read
 *   only), state_bytes >= tpk_gdn_workspace_bytes.
 *   workspace: >= tpk_gdn_bwd_workspace_bytes bytes, 256-byte aligned, need
 *   not be cleared: the initial-state gradients (n_seg_instances * H * dk * dv
 *   fp32) and, reused level by level, each chain's checkpoints (its state
 *   every 32 tokens) and per-token values (u_t, S_{t-1} k_t, 1/|k_t|,
 *   do_t . o_t), sized by the largest level.
 * Outputs may be column slices of one [F, ld] tensor (the convolution's
 * gradient), with 16-byte aligned rows.  TPK_E_UNSUPPORTED for other head
 * sizes, TPK_E_ARG for bad pointers or strides, TPK_E_WORKSPACE for a short
 * or misaligned workspace. */
size_t tpk_gdn_bwd_workspace_bytes(const tpk_plan* plan, int32_t H, int32_t dk, int32_t dv);
int tpk_gdn_delta_rule_bwd(const tpk_plan* plan, const void* dev_image, const void* q, const void* k,
                           const void* v, int64_t ld_qk, int64_t ld_v, const float* g, const float* beta,
                           const void* dout, void* dq, void* dk_, void* dv_, int64_t ld_dqk, int64_t ld_dv,
                           float* dg, float* dbeta, int32_t H, int32_t dk, int32_t dv, float scale,
                           const void* state, size_t state_bytes, void* workspace, size_t ws_bytes, void* stream);

/* Self-test of the device-side failure path (no counterpart on the pages):
 * launches one small kernel that waits, with the same bounded mbarrier wait
 * the attention kernels use, on a barrier nothing ever arrives at.  After
 * limit_ns nanoseconds (1 .. 2e9) the wait gives up, TPK_E_TIMEOUT is written
 * to *dev_err (device int32) and the kernel exits; the context stays usable.
 * Used by the tests to check timeout reporting without faulting or hanging
 * the GPU. */
int tpk_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_err, void* stream);

const char* tpk_status_string(int status);

/* Library version string. */
const char* tpk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPK_H_ */
