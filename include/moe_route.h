/*
 * moe_route.h -- C ABI of the GB300 fused mixture-of-experts layer forward.
 *
 * The library computes, for T tokens, E experts and top-k routing:
 *   a-1  NaN-safe softmax / sigmoid top-k routing with k distinct ids
 *        (PR #39593 "Fix FlashInfer CUTLASS BF16 + CUDA graphs IMA",
 *        section "Fix": NaN replaced by -FLT_MAX in-register before scoring
 *        and before the arg-max, so that top-k yields k distinct ids),
 *   a-2  count and permute token rows by expert (H20 article, para. 3: the
 *        rows each expert receives),
 *   a-3  the tile plan from the rows-per-expert estimate
 *        est = max(1, ceil(T*k/E)), applied after the worst-case workspace
 *        capacity is fixed (H20 article, para. 3),
 *   a-4  grouped gate+up GEMM, a-5 SiLU(gate)*up, a-6 grouped down GEMM,
 *   a-7  the top-k weighted combine back to token order
 *        (H20 article, para. 2: fused expert computations with FP8 block
 *        scaling; Lab notes #6, "Method": fp8_w8a8, block [128,128]).
 *
 * Conventions for every call:
 *  - Every pointer argument named "device" is a device pointer the caller
 *    owns (e.g. from torch); the library never allocates device memory and
 *    keeps no state beyond a per-device cache of kernel attributes and a
 *    cache of TMA tensor maps keyed by device, pointers and shapes (a map
 *    encodes only an address, a shape and a box, so an entry stays valid
 *    while the same pointers come with the same shapes).
 *  - `stream` is a cudaStream_t passed as void*; all device work is
 *    enqueued on it asynchronously.  No call below synchronises, except
 *    moe_check.
 *  - Every call returns MOE_OK (0) or a negative MOE_ERR_* code.  Argument
 *    and shape validation happens before any launch; nothing is enqueued
 *    when an argument is rejected.
 *  - Layouts are row-major (C order).  "flat index" f = t*k + j, where j is
 *    the rank of the pick within token t (0 = highest scored).
 *
 * Weights:  w13 [E, 2I, H]: rows [0, I) are the gate projection and rows
 *           [I, 2I) the up projection of each expert; w2 [E, H, I].
 *  MOE_DTYPE_F32:  x [T,H] f32, logits [T,E] f32, w13/w2 f32, out [T,H]
 *                  f32.  GEMMs run on the tensor cores as TF32.
 *  MOE_DTYPE_BF16: x, logits, w13, w2 and out in bf16.
 *  MOE_DTYPE_FP8_BLOCK128: x and logits bf16; w13 / w2 are e4m3 codes with
 *                  fp32 block scales s13 [E, 2I/128, H/128] and
 *                  s2 [E, H/128, I/128] (one scale per [128,128] block);
 *                  activations are quantised inside the call per token and
 *                  128-column group (scale = max(amax,1e-10)/448, clamp
 *                  fmaxf(fminf(v,448),-448), round to nearest even);
 *                  out bf16.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

/* return codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* null pointer, bad size, bad enum, misaligned pointer */
#define MOE_ERR_UNSUPPORTED (-2) /* valid but not supported (e.g. FP8 with H % 128 != 0) */
#define MOE_ERR_WORKSPACE (-3)   /* ws_bytes smaller than plan->workspace_bytes */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed */
#define MOE_ERR_DEVICE (-5)      /* moe_check: the device error word is set */
#define MOE_ERR_TIMEOUT (-6)     /* moe_check: a device wait gave up */

/* device error word bits (moe_check) */
#define MOE_DEVERR_BAD_ID 1u   /* a caller-supplied id outside [0, E) (skipped) */
#define MOE_DEVERR_DUP_ID 2u   /* a caller-supplied id repeated within a token (skipped) */
#define MOE_DEVERR_TIMEOUT 4u  /* a pipeline wait exceeded its limit; kernel returned */
#define MOE_DEVERR_CAPACITY 8u /* tile list would exceed the planned capacity */

/* compute dtypes */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1
#define MOE_DTYPE_FP8_BLOCK128 2

/* logits dtypes (moe_route_topk) */
#define MOE_LOGITS_F32 0
#define MOE_LOGITS_BF16 1

/* scoring */
#define MOE_SCORING_SOFTMAX 0
#define MOE_SCORING_SIGMOID 1

/*
 * The plan: pure host arithmetic, filled by moe_plan.  All offsets are
 * byte offsets into the caller's workspace, 256-byte aligned, so that tests
 * can read the intermediates:
 *   ids     int32 [T, k]    chosen expert per pick (-1 = skipped, see with_ids)
 *   w       f32   [T, k]    combine weight per pick
 *   counts  int32 [e_local] rows per (local) expert
 *   offsets int32 [e_local + 1] exclusive scan of counts
 *   src     int32 [T*k]     permuted row -> flat index (expert-major,
 *                           ascending flat index within an expert)
 *   pos     int32 [T*k]     flat index -> permuted row (inverse of src)
 *   tiles   int32 [max_tiles, 4]  {expert, first row, rows, width} token
 *                           tiles of grouped GEMM 1, in expert order (CTA-pair
 *                           plans: experts that fill a whole 256-row tile
 *                           first, then the rest, each group in expert order)
 *   ntiles  int32 [1]       number of valid tiles
 *   tiles2, ntiles2         the same for grouped GEMM 2 when its widths differ
 *                           (prefill-sized BF16/F32 plans); otherwise unused
 *   dep     int32 [max_tiles + 2] finished GEMM1 items per tile (when both
 *                           GEMMs run as one launch), then the work counters
 *                           of the GEMM launches
 *   err     uint32 [1]      device error word (MOE_DEVERR_* bits); the two
 *                           words after it are internal: the call's routing
 *                           breadth (read by the next call on the same
 *                           workspace to decide an early weight prefetch),
 *                           and the GEMM kernel family the call chose (1 one
 *                           CTA per tile, 2 CTA pairs; see gemm_dyn)
 *   y       [T*k, H]        routing-weighted expert output per permuted
 *                           row (bf16; f32 for the f32 layer)
 * The remaining regions (chunk counts, permuted activations, scales) are
 * internal.
 */
typedef struct moe_plan {
  int32_t abi_version;
  int32_t T, H, I, E, k;
  int32_t dtype, scoring, renorm;
  int32_t est;        /* rows-per-expert estimate used for the tile choice */
  int32_t force_est;  /* 0, or the caller's override (e.g. T: old estimate) */
  int32_t tile_n;     /* token tile (16, 32, 64 or 128; FP8 at most 64) from
                         est; the device widens it per expert for BF16/F32 (an
                         expert with more rows gets 32 / 64 / 128, for grouped
                         GEMM 2 256 when est > 64, and up to 256 for both GEMMs
                         in CTA-pair plans).  The MMAs of a tile compute its
                         rows rounded up to 16. */
  int32_t route_tpc;  /* tokens per routing CTA */
  int32_t n_chunks;   /* routing CTAs = ceil(T / route_tpc) */
  int32_t max_tiles;  /* worst-case token tiles (independent of est) */
  int32_t g1_mblocks; /* ceil(I / 128) gate+up feature blocks (CTA pairs take
                         256 features per work item) */
  int32_t g2_mblocks; /* ceil(H / 128) output feature blocks (CTA pairs: 256) */
  int32_t ep_size;    /* expert-parallel ranks (1: all experts local) */
  int32_t ep_rank;    /* this rank; it holds experts [ep_rank*e_local, +e_local) */
  int32_t e_local;    /* E / ep_size: experts in w13/w2/s13/s2 of this call */
  int32_t n_group;    /* group-limited routing: expert groups (1 = off) */
  int32_t topk_group; /* groups kept per token */
  int32_t gemm_pair;  /* 1: the grouped GEMMs run on CTA pairs (cta_group::2,
                         BF16/F32 with est > 32): token tiles up to 256 rows,
                         items of 256 weight rows; 0: one CTA per tile (but
                         see gemm_dyn).  Set by moe_plan; a caller may clear
                         or set it (ignored for FP8). */
  int32_t gemm_tm;    /* FP8 only.  1: token-major grouped GEMMs -- every
                         expert's rows in tiles of 128 on the MMA's M side,
                         256 weight rows on its N side (gate and up rows of a
                         128-feature block for GEMM 1, two 128-row blocks of
                         w2 for GEMM 2); 0: weight rows on the M side and
                         token tiles of tile_n.  Set by moe_plan when
                         est >= 32; a caller may clear or set it. */
  int32_t gemm_dyn;   /* BF16/F32 plans with gemm_pair 0.  1: the device picks
                         the kernel family per call -- CTA pairs when an
                         expert holds 256 rows or more (concentrated routing,
                         which the estimate does not foresee), one CTA per
                         tile otherwise; both families' launches are queued
                         and those of the family not picked return at once.
                         Set by moe_plan when est <= 32 and T >= 256; a
                         caller may clear it (setting it on another plan has
                         no effect). */
  uint64_t workspace_bytes;
  uint64_t off_err, off_ids, off_w, off_chunk_counts, off_lrank, off_counts, off_offsets;
  uint64_t off_chunk_base, off_src, off_pos, off_tiles, off_ntiles;
  uint64_t off_xq, off_xs, off_act, off_as, off_y;
  uint64_t off_tiles2, off_ntiles2, off_dep;
  uint64_t reserved1[1];
} moe_plan_t;

/*
 * moe_plan -- fill *plan for one layer shape.  Pure host arithmetic; no
 * device call.  Requirements: T >= 0; 1 <= E <= 1024; 1 <= k <= min(E, 32);
 * H, I multiples of 32 (F32), 64 (BF16) or 128 (FP8); scoring softmax or
 * sigmoid.  The workspace capacity is fixed first from (T, k, E, H, I,
 * dtype) alone; then est = force_est if force_est > 0, else
 * max(1, ceil(T*k/E)), and tile_n = 16 / 32 / 64 / 128 for est <= 16 /
 * <= 32 / <= 64 / above (FP8: at most 64, the width its scale-folding
 * epilogue holds in registers).
 * Errors: MOE_ERR_INVALID_ARG (null plan, negative or out-of-range sizes,
 * bad enums), MOE_ERR_UNSUPPORTED (H or I not a multiple of the dtype's
 * K step).
 */
int moe_plan(int T, int H, int I, int E, int k, int dtype, int scoring, int renorm, int force_est,
             moe_plan_t* plan);

/*
 * moe_plan_ep -- moe_plan for one expert-parallel rank (H20 article,
 * para. 2: the fused-MoE API takes the expert-parallel size and rank).  E is
 * the number of experts over all ranks (E % ep_size == 0); this rank holds
 * experts [ep_rank*E/ep_size, (ep_rank+1)*E/ep_size), and w13/w2/s13/s2
 * passed with this plan hold only those e_local = E/ep_size experts.
 * Routing ranks all E experts (logits [T, E]); picks of other ranks'
 * experts are skipped, so out is this rank's partial sum -- the layer's
 * output is the sum over ranks (the exchange between ranks is the caller's).
 * The estimate divides by all E experts.  counts/offsets/tiles use local
 * expert indices; ids keep the global ones.  moe_plan is moe_plan_ep with
 * ep_size 1, ep_rank 0.  Errors as moe_plan, and MOE_ERR_INVALID_ARG for a
 * bad ep_size / ep_rank.
 */
int moe_plan_ep(int T, int H, int I, int E, int k, int dtype, int scoring, int renorm,
                int force_est, int ep_size, int ep_rank, moe_plan_t* plan);

/*
 * moe_plan_set_groups -- switch a plan to group-limited routing: the E
 * experts form n_group contiguous groups of E/n_group; a token keeps the
 * topk_group groups with the largest sanitised logit (ties to the lower
 * group) and picks its top-k among their experts only.  PR #39593 ("Test
 * Plan") requires this grouped top-k, too, to return distinct experts for
 * all-NaN rows; the pages do not define the grouping itself, and the group
 * score used here (the group's best logit) is the plainest reading.
 * Requires n_group <= 32, E % n_group == 0, 1 <= topk_group <= n_group and
 * k <= topk_group * E / n_group; else MOE_ERR_INVALID_ARG.  Host only.
 */
int moe_plan_set_groups(moe_plan_t* plan, int n_group, int topk_group);

/*
 * moe_forward -- steps a-1 .. a-7 for one batch, asynchronously on stream.
 *   x       device, [T, H] (f32 for F32, else bf16)
 *   logits  device, [T, E] gating logits (f32 for F32, else bf16); NaN and
 *           +-Inf allowed (NaN -> -FLT_MAX, +-Inf -> +-FLT_MAX)
 *   w13     device, [E, 2I, H]; w2 device, [E, H, I] (dtype per plan)
 *   s13,s2  device fp32 block scales for FP8, else must be NULL
 *   out     device, [T, H] (f32 for F32, else bf16); fully overwritten
 *   ws      device workspace of ws_bytes >= plan->workspace_bytes
 * x, w13, w2, out and ws must be 16-byte aligned.  T == 0 enqueues nothing
 * and accepts null activation, output and workspace pointers.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
int moe_forward(const moe_plan_t* plan, const void* x, const void* logits, const void* w13,
                const float* s13, const void* w2, const float* s2, void* out, void* ws,
                size_t ws_bytes, void* stream);

/*
 * moe_forward_timed -- moe_forward that also records caller-created CUDA
 * events (cudaEvent_t passed as void*) on `stream` at the boundaries of its
 * launches, for per-kernel timing without a profiler: events[0] before the
 * routing kernel, [1] after routing, [2] after the scan, [3] after the
 * gather, [4] after grouped GEMM 1, [5] after grouped GEMM 2, [6] after the
 * combine.  When both GEMMs run as one launch, [4] follows that launch and
 * [5] directly follows [4].  When the device chooses the kernel family (see
 * gemm_dyn), [4] follows the one-CTA-per-tile launch and [5] the CTA-pair
 * launches; the launches of the family not chosen do no work.  n_events must be 7.  Same
 * arguments, errors and results as moe_forward otherwise.
 */
int moe_forward_timed(const moe_plan_t* plan, const void* x, const void* logits, const void* w13,
                      const float* s13, const void* w2, const float* s2, void* out, void* ws,
                      size_t ws_bytes, void* stream, void* const* events, int n_events);

/*
 * moe_forward_with_ids -- as moe_forward, but routing (a-1) is replaced by
 * caller-supplied ids (device int32 [T, k]) and weights (device f32
 * [T, k]).  Each pick is validated on the device: an id outside [0, E), or
 * repeated within its token, sets MOE_DEVERR_BAD_ID / MOE_DEVERR_DUP_ID in
 * the error word and that pick is skipped (contributes nothing) instead of
 * being used as an index.  This is the fault-test entry for the
 * duplicate-id failure described in PR #39593 ("Root cause").
 */
int moe_forward_with_ids(const moe_plan_t* plan, const void* x, const int32_t* ids,
                         const float* topk_w, const void* w13, const float* s13, const void* w2,
                         const float* s2, void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_route_topk -- step a-1 alone: logits (device [T, E], MOE_LOGITS_*)
 * -> ids (device int32 [T, k]) and w (device f32 [T, k]).  Selection is on
 * the sanitised logits, descending, ties to the lower expert index; softmax
 * weights are exp(l - max) / sum over all E, sigmoid weights 1/(1+exp(-l));
 * renorm != 0 rescales the k weights to sum to one (1/k each when their sum
 * is zero or not finite).  Requires 1 <= E <= 1024, 1 <= k <= min(E, 32).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
int moe_route_topk(const void* logits, int logits_dtype, int T, int E, int k, int scoring,
                   int renorm, int32_t* ids, float* w, void* stream);

/*
 * moe_route_grouped_topk -- moe_route_topk with group-limited selection
 * (see moe_plan_set_groups); n_group 1 is moe_route_topk.
 */
int moe_route_grouped_topk(const void* logits, int logits_dtype, int T, int E, int k,
                           int n_group, int topk_group, int scoring, int renorm, int32_t* ids,
                           float* w, void* stream);

/*
 * moe_check -- synchronise `stream`, read the workspace error word, clear
 * it, and return MOE_OK, MOE_ERR_TIMEOUT (timeout bit set) or
 * MOE_ERR_DEVICE (any other bit).  *bits (if not NULL) receives the word.
 */
int moe_check(const moe_plan_t* plan, void* ws, uint32_t* bits, void* stream);

/* moe_plan_describe -- a one-line text summary of the plan (est, tile,
 * workspace) into buf (NUL-terminated, truncated to n).  Returns the
 * length it wanted, or MOE_ERR_INVALID_ARG. */
int moe_plan_describe(const moe_plan_t* plan, char* buf, size_t n);

/*
 * moe_forward_noalloc -- moe_forward for callers that cannot allocate
 * device memory (code running inside an allocator hook or a memory pool,
 * plug-ins whose host forbids device allocation after start-up, call sites
 * that must run in a fixed memory budget).  The pages have no counterpart of
 * this entry point.
 *
 * The workspace is a 16 MiB array inside the library's device image
 * (reserved on every GPU that loads the library, held until the process
 * exits); nothing is allocated, by this call or by the library.  Plans whose
 * workspace_bytes exceed 16 MiB are rejected with MOE_ERR_WORKSPACE before
 * any launch (for example T=128, H=2048, I=768, E=128, k=8 in bf16 needs
 * about 10 MB).  The caller still passes inputs and outputs, with the same
 * layouts, alignment and errors as moe_forward.
 *
 * The first call on each device looks up the array's device address
 * (a synchronous runtime query, with that device current); make that first
 * call before any stream capture.  The address is looked up again when the
 * device's context changes (after cudaDeviceReset, for example), and that
 * next call is again a first call.  Every call on a device uses the same
 * array and leaves its contents behind; the call clears what must start at
 * zero itself.  Calls whose work overlaps on the GPU (other streams, other
 * threads) race on the array: serialise them.  The device error word lives
 * in that array; read it with moe_check_noalloc.
 */
int moe_forward_noalloc(const moe_plan_t* plan, const void* x, const void* logits,
                        const void* w13, const float* s13, const void* w2, const float* s2,
                        void* out, void* stream);

/*
 * moe_check_noalloc -- moe_check for moe_forward_noalloc: synchronise
 * `stream`, read and clear the error word in the built-in workspace of the
 * current device (at plan->off_err), and return MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE as moe_check does; *bits (if not NULL) receives the word.
 * Allocates nothing.  MOE_ERR_WORKSPACE for a plan too large for the
 * built-in workspace; MOE_ERR_INVALID_ARG for a bad plan.  The pages have no
 * counterpart of this call either.
 */
int moe_check_noalloc(const moe_plan_t* plan, uint32_t* bits, void* stream);

/*
 * Expert parallelism across ranks (H20 article, para. 2: the fused-MoE call
 * takes the expert-parallel size and rank; para. 3: 400 expert slots over
 * 8 GPUs).  Each rank routes its own T tokens over all E = e_local * ep_size
 * experts, sends every token once to each rank that owns at least one of its
 * picks (owner = id / e_local), runs moe_forward_with_ids on an
 * expert-parallel plan (moe_plan_ep) over the rows it receives, and sums the
 * partial rows that come back.  The three calls below are that exchange's
 * arithmetic; moving rows between ranks (an all-to-all) is the caller's.
 * They are asynchronous on `stream` and allocate nothing; ep_size <= 32.
 *
 * moe_ep_dispatch -- the send plan.
 *   ids          device int32 [T, k] global expert ids (picks outside
 *                [0, E) are ignored)
 *   send_counts  device int32 [ep_size] out: tokens sent to each rank
 *   send_tokens  device int32 [T * ep_size] out: the sent tokens, grouped by
 *                destination rank in rank order, each group in token order
 *                (entries past the total are left as they were)
 *   row_of       device int32 [T, ep_size] out: the send row of (token,
 *                rank), or -1 when the token is not sent to that rank
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
int moe_ep_dispatch(const int32_t* ids, int T, int k, int e_local, int ep_size,
                    int32_t* send_counts, int32_t* send_tokens, int32_t* row_of, void* stream);

/*
 * moe_ep_pack -- gather the send rows of moe_ep_dispatch's plan: send row r
 * (r below the total of send_counts) receives token send_tokens[r]'s
 * activation row (x [T, H], MOE_DTYPE_F32 or MOE_DTYPE_BF16), its k ids and
 * its k weights (w device f32 [T, k]).  x_send [T * ep_size, H], ids_send
 * [T * ep_size, k] and w_send [T * ep_size, k] are the caller's buffers;
 * rows past the total are not written.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
int moe_ep_pack(const void* x, int x_dtype, const int32_t* ids, const float* w, int T, int H,
                int k, int ep_size, const int32_t* send_counts, const int32_t* send_tokens,
                void* x_send, int32_t* ids_send, float* w_send, void* stream);

/*
 * moe_ep_combine -- the layer's output from the partial rows that came back
 * (back device f32 [n, H], row r the owner's partial sum for send row r):
 * out[t] = sum over d = 0, 1, ..., ep_size-1 with row_of[t, d] >= 0 of
 * back[row_of[t, d]], added in that (rank) order, so the result does not
 * depend on arrival order; a token with no row gets zeros.  out device f32
 * [T, H].  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
int moe_ep_combine(const float* back, const int32_t* row_of, int T, int H, int ep_size,
                   float* out, void* stream);

/* moe_strerror -- static message for a MOE_* return code. */
const char* moe_strerror(int code);

/* moe_abi_version -- MOE_ABI_VERSION of the built library. */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
