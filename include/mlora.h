/*
 * mlora.h — C ABI of the packed multi-adapter LoRA layer (forward, backward, AdamW).
 *
 * Many LoRA jobs share one frozen base weight W (d_in x d_out).  Job i owns a
 * contiguous run of token rows X_i (rows [tok_offset_i, tok_offset_i + n_i) of
 * the packed activation X, N x d_in), a rank r_i, a scale s_i = alpha_i / r_i and
 * trainable A_i (d_in x r_i), B_i (r_i x d_out).  The layer computes
 *
 *     Y_i  = X_i W + s_i (X_i A_i) B_i                              (forward)
 *     H_i  = X_i A_i                                                (saved activation)
 *     dH_i = s_i dY_i B_i^T,   dB_i = s_i H_i^T dY_i                (B-side gradients)
 *     dA_i = X_i^T dH_i,       dX_i = dY_i W^T + dH_i A_i^T         (A-side gradients)
 *
 * followed by one decoupled-weight-decay AdamW step on every A_i and B_i.
 *
 * Sources: "PLoRA: Efficient Concurrent LoRA Training for Large Language
 * Models" (full text), §2.1 (the LoRA layer: A is d x r, B is r x k), §2.4
 * (packing: every job applies its own adapter to its own inputs), §9.2
 * "Packed LoRA Kernels" (the four backward products, Cases 1-4, and the rule
 * that tiles run along the token or hidden dimensions, never along the rank),
 * §8 (AdamW keeps gradient, first and second moment per parameter).  "tLoRA:
 * Efficient Multi-LoRA Training with Elastic Shared Super-Models" (abstract)
 * for the rank-aware grouping of uneven jobs into one launch.
 *
 * Storage (all row-major, all device pointers unless stated):
 *   X   [N, d_in]      bf16 (MLORA_BF16) or fp32 (MLORA_F32)
 *   Wt  [d_out, d_in]  W transposed, same dtype as X (the nn.Linear weight layout)
 *   Y   [N, d_out], dY [N, d_out], dX [N, d_in]: same dtype as X
 *   At_i [r_i, d_in], Bt_i [d_out, r_i]: fp32 masters (A_i, B_i transposed);
 *   dAt_i, dBt_i, mA_i, vA_i, mB_i, vB_i: fp32, same shapes as At_i / Bt_i.
 *   H, dH: fp32, job i's [n_i, r_i] block stored row-major at element offset
 *          sum_{j<i} n_j r_j (mlora_h_elems() gives the total).
 * Ownership: the caller allocates and frees every buffer named above, the
 * workspace and the stream.  A plan owns only its own small device tables
 * (segment table, tile lists, status word) and a copy of the segment table.
 * Every call is asynchronous on the given stream (a cudaStream_t passed as
 * void*; NULL = legacy default stream) and returns an error code at once for
 * anything detectable on the host; nothing crosses the ABI as an exception.
 * A device-side wait that gives up (see MLORA_ERR_TIMEOUT) records its code in
 * the plan's status word, read back by mlora_sync_status().
 * Threads: different plans may be used from different host threads at once (each call makes
 * the plan device's primary context current on its thread); calls on one plan must not overlap
 * on the host, and their launches must not run at the same time on the device either (one
 * stream, or streams ordered by events): a plan's status word and the arrival counters of its
 * work items that are cut across CTAs belong to the plan.  mlora_forward, mlora_backward and
 * mlora_adamw (and their _w4 / _ws forms) can be captured into a CUDA graph.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mlora_status {
    MLORA_OK = 0,
    MLORA_ERR_INVALID = 1,      /* bad argument: null pointer, bad segment table, misaligned buffer */
    MLORA_ERR_UNSUPPORTED = 2,  /* valid but outside what this library implements (e.g. rank > 256) */
    MLORA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed; mlora_last_error() has the text */
    MLORA_ERR_TIMEOUT = 4,      /* a device-side wait gave up (reported by mlora_sync_status) */
    MLORA_ERR_OOM = 5           /* the plan's small device tables could not be allocated */
} mlora_status;

typedef enum mlora_dtype {
    MLORA_F32 = 0,     /* X, W, dY, Y, dX in fp32; true fp32 FFMA arithmetic */
    MLORA_BF16 = 1,    /* X, W, dY, Y, dX in bf16; tensor-core products with fp32 accumulation */
    MLORA_BF16_W4 = 2  /* X, dY, Y, dX in bf16, the frozen W as 4-bit codes with fp32 group scales
                          (mlora_forward_w4 / mlora_backward_w4); d_in a multiple of 64 */
} mlora_dtype;

/* mlora_problem.flags */
#define MLORA_PLAN_HOST_ONLY 1u        /* build and validate the tables on the host only: no CUDA call,
                                          the plan can be inspected but not executed */
#define MLORA_DEBUG_SHORT_TIMEOUT 2u   /* device waits give up after ~1 ms instead of ~4 s */
#define MLORA_DEBUG_DROP_COPY 16u      /* test hook, honoured only with MLORA_DEBUG_SHORT_TIMEOUT: in the
                                          forward's first tensor-core launch one CTA arms a pipeline slot
                                          but copies nothing into it, so a device wait runs out (~1 ms),
                                          the status word records it and mlora_sync_status() returns
                                          MLORA_ERR_TIMEOUT; that call's outputs are undefined */
#define MLORA_DEBUG_DROP_COPY_PAIRS 512u  /* test hook, honoured only with MLORA_DEBUG_SHORT_TIMEOUT: in the
                                          forward's CTA-pair kernels (the shrink when it runs on pairs, and
                                          the base GEMM) the first pair's even CTA arms its first pipeline
                                          slot for both CTAs' bytes but copies nothing into it; the MMA's
                                          wait runs out (~1 ms), each kernel drains its peer's copies and
                                          returns, and mlora_sync_status() returns MLORA_ERR_TIMEOUT; that
                                          call's outputs are undefined */
#define MLORA_REUSE_STAGING 32u       /* mlora_backward skips rebuilding the bf16 adapter shadows and the
                                          staged s*H images when its workspace and H are the ones the last
                                          mlora_forward of this plan used and no AdamW step ran since (and,
                                          for a 4-bit base, the bf16 expansion of W when Wq and Wscale are the
                                          forward's pointers); mlora_forward skips rebuilding the shadows when
                                          its workspace holds them for the current masters (left by the last
                                          forward or backward with no AdamW step since, or refreshed by
                                          mlora_adamw_ws).  The caller guarantees that neither At/Bt, H,
                                          Wq/Wscale nor that workspace changed in between except through
                                          these calls (results are then identical to the full passes) */
#define MLORA_NO_OVERLAP 8u            /* launch every kernel strictly after the previous one (no programmatic
                                          dependent launch overlapping a kernel's prologue with the tail of
                                          the one before); results are identical either way.  Plans whose
                                          base product n_tokens * d_in * d_out exceeds 4e11 launch this way
                                          by default (measured faster there) */
#define MLORA_OVERLAP 1024u           /* keep the programmatic overlap whatever the plan's size (MLORA_NO_OVERLAP
                                          wins if both are given) */
#define MLORA_GEMM_SINGLE_CTA 4u       /* run the two base GEMMs on single-CTA 128x256 tiles instead of
                                          CTA pairs (256x256 tiles); same results up to rounding order */
#define MLORA_WINDOW_PAIRS 128u        /* run the shrink and dH products on CTA pairs (256-token tiles sharing
                                          the rank operand, up to four 64-column chunks per item) whatever
                                          the planner would pick; same results up to rounding order */
#define MLORA_WINDOW_SINGLE 256u       /* run them on the single-CTA engine (128-token tiles, two chunks per
                                          item).  Without either flag the planner takes pairs when the
                                          token tiles' rank windows average more than 1.25 chunks */
#define MLORA_W4_FUSED 64u             /* 4-bit base only: expand the codes to bf16 inside the CTA-pair base
                                          GEMMs (converter warps, once per 256-token tile pair) instead of
                                          once per call into the workspace; the workspace is smaller by
                                          2 d_in d_out bytes, the GEMMs slower when the pack spans many
                                          tile pairs; identical results; not with MLORA_GEMM_SINGLE_CTA */

/* One job of the pack.  Pointers are device pointers to fp32 buffers of the
 * shapes given above, each 16-byte aligned.  dAt/dBt are overwritten (not
 * accumulated) by mlora_backward; At/Bt/mA/vA/mB/vB are updated in place by
 * mlora_adamw.  Pointers unused by a call may be NULL for that call only if
 * the plan was built with them NULL (e.g. a forward-only plan). */
typedef struct mlora_segment {
    int64_t tok_offset;   /* first row of this job in X / dY / Y / dX */
    int32_t n_tokens;     /* n_i >= 1 */
    int32_t rank;         /* 1 <= r_i <= 256 */
    float scale;          /* s_i = alpha_i / r_i */
    float* At;
    float* Bt;
    float* dAt;
    float* dBt;
    float* mA;
    float* vA;
    float* mB;
    float* vB;
} mlora_segment;

typedef struct mlora_problem {
    int64_t n_tokens;     /* N: rows of X; the segments must tile [0, N) in order, without gaps */
    int32_t d_in;         /* multiple of 8 (bf16) or 4 (fp32) */
    int32_t d_out;        /* multiple of 8 (bf16) or 4 (fp32) */
    int32_t dtype;        /* mlora_dtype */
    uint32_t flags;       /* MLORA_PLAN_* / MLORA_DEBUG_* bits */
    int64_t mem_budget_bytes;  /* 0: no check.  Otherwise the device memory this layer may use: the
                                  plan is refused with MLORA_ERR_OOM when mlora_memory_estimate's
                                  total exceeds it (PLoRA §8: M_base + sum_k M_lora,k must stay
                                  within c_load x M_gpu; the caller passes its share for this layer) */
} mlora_problem;

typedef struct mlora_plan_s mlora_plan_t;

/* Validate the segment table and build the tile schedule (the M-tile to job
 * map, the per-tile rank windows and the rank-aware work lists of every
 * kernel), then upload it to the current device.  On success *out is a plan
 * that stays valid, immutable and reusable for any number of steps while the
 * shapes and the segment table's pointers stay the same, and
 * *workspace_bytes is the size of the scratch buffer that forward/backward
 * need (caller-allocated device memory, 256-byte aligned, contents need not
 * be initialised).  Errors: MLORA_ERR_INVALID (null/misaligned pointers,
 * segments out of order, overlapping, leaving gaps, n_i < 1, bad dims),
 * MLORA_ERR_UNSUPPORTED (rank > 256, d not a multiple of 8/4),
 * MLORA_ERR_OOM / MLORA_ERR_CUDA (device tables). */
mlora_status mlora_plan(const mlora_problem* problem, const mlora_segment* segs, int32_t n_segs,
                        size_t* workspace_bytes, mlora_plan_t** out);

/* Shared-input pack: several projections read the same input X (the q, k and v projections of
 * an attention block, or gate and up of an MLP), and each job trains one adapter per
 * projection.  Their frozen weights are stacked into one W^T [d_out, d_in] whose output columns
 * fall into n_groups groups, group g covering [col_offset_g, col_offset_g + d_out_g) (the
 * groups tile [0, d_out) in order), and Y = X W is the projections' outputs side by side.
 * ("PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §8 names the seven
 * adaptable projections of a block; sharing their input across one pass over X is this
 * library's design, the pages describe no such kernel.)
 *
 * segs holds n_jobs x n_groups entries, job-major: segs[j * n_groups + g] is job j's adapter
 * on group g, with Bt [d_out_g, r] (its own group's columns only; dBt, mB, vB alike) and
 * At [r, d_in]; all entries of a job give the same tok_offset and n_tokens, and the jobs tile
 * [0, N) in order.  Each adapter computes exactly what a one-group plan would on its group:
 *     Y_j[:, group g] = X_j W_g + s_jg (X_j A_jg) B_jg,
 *     dX_j = dY_j W^T + sum_g s_jg dY_j[:, group g] B_jg^T A_jg^T,
 * with its own gradients and AdamW state.  H and dH hold job j's block [n_j, R_j] at element
 * offset sum_{i<j} n_i R_i, R_j = sum_g r_jg, adapter g in columns [sum_{h<g} r_jh, ... + r_jg).
 * One pass over X computes every adapter's H (and one pass over dY every dH).  bf16 and 4-bit
 * bases only (MLORA_ERR_UNSUPPORTED for fp32 with more than one group); otherwise errors,
 * ownership and the entry points are those of mlora_plan, which is this call with one group
 * {0, d_out}. */
typedef struct mlora_group {
    int32_t col_offset;   /* first output column of the group in Y / dY / rows of W^T */
    int32_t d_out;        /* its width (>= 1) */
} mlora_group;

mlora_status mlora_plan_grouped(const mlora_problem* problem, const mlora_group* groups, int32_t n_groups,
                                const mlora_segment* segs, int32_t n_segs, size_t* workspace_bytes,
                                mlora_plan_t** out);

/* Free the plan's device tables (after work using it has finished). NULL is a no-op. */
void mlora_plan_destroy(mlora_plan_t* plan);

/* Forward pass: Y = X W + s_i (X_i A_i) B_i per job, and the saved activation
 * H (fp32, packed as described above).  Reads At_i/Bt_i of every segment. */
mlora_status mlora_forward(const mlora_plan_t* plan, const void* X, const void* Wt, void* Y, float* H,
                           void* workspace, void* stream);

/* 4-bit base ("PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §5 and
 * §11.3: a QLoRA-quantised base composes with packing; the pages do not fix the format).
 * For plans of dtype MLORA_BF16_W4 the frozen W is given as
 *   Wq     [d_out, d_in / 2] bytes: the signed 4-bit code q[o][k] in [-8, 7] of W[k][o], two per
 *          byte, even k in the low nibble (two's complement);
 *   Wscale [d_in / 64, d_out] fp32: one scale per 64 consecutive k of each output column;
 * and the layer uses W[k][o] = bf16(q[o][k] * Wscale[k / 64][o]) (the product in fp32, rounded
 * to nearest bf16), which is what the bf16 entry points would compute with that Wt.  Unless the
 * plan has MLORA_W4_FUSED, each call first expands W into the workspace as bf16 Wt (which is
 * why the workspace of such a plan holds 2 d_in d_out more bytes) and then runs the bf16 path.
 * Everything else (arguments, layouts, errors) is as for mlora_forward / mlora_backward.  Both
 * pointers 16-byte aligned. */
mlora_status mlora_forward_w4(const mlora_plan_t* plan, const void* X, const void* Wq, const float* Wscale,
                              void* Y, float* H, void* workspace, void* stream);
mlora_status mlora_backward_w4(const mlora_plan_t* plan, const void* X, const void* Wq, const float* Wscale,
                               const void* dY, const float* H, void* dX, float* dH, void* workspace,
                               void* stream);

/* Backward pass given the upstream gradient dY and the forward's H:
 * writes dX, dH (fp32, packed like H) and every segment's dAt/dBt. */
mlora_status mlora_backward(const mlora_plan_t* plan, const void* X, const void* Wt, const void* dY,
                            const float* H, void* dX, float* dH, void* workspace, void* stream);

/* One AdamW step on every job's A and B (PyTorch's order: decay p by
 * (1 - lr*weight_decay), update the moments, bias-correct with step t >= 1,
 * then p -= lr * m_hat / (sqrt(v_hat) + eps)).  Reads dAt/dBt; updates
 * At/Bt/mA/vA/mB/vB in place.  Moments start at zero at t = 1 (caller-zeroed). */
mlora_status mlora_adamw(const mlora_plan_t* plan, float lr, float beta1, float beta2, float eps,
                         float weight_decay, int32_t step, void* stream);

/* mlora_adamw that also writes the updated A_i, B_i into the bf16 shadows held in `workspace`
 * (the copies the kernels read, rounded as a fresh pack would round them), so that the next
 * mlora_forward with that workspace under MLORA_REUSE_STAGING starts without rebuilding them.
 * The shadows count as current only if a forward or backward built them in this workspace
 * before (their zero padding is not rewritten); otherwise the next forward rebuilds them.
 * fp32 plans have no shadows: this is mlora_adamw.  Errors as mlora_adamw, plus MLORA_ERR_INVALID
 * for a null or misaligned workspace. */
mlora_status mlora_adamw_ws(const mlora_plan_t* plan, float lr, float beta1, float beta2, float eps,
                            float weight_decay, int32_t step, void* workspace, void* stream);

/* Synchronise the stream, then read and clear the plan's device status word:
 * MLORA_OK, or MLORA_ERR_TIMEOUT if a device-side wait gave up since the last
 * call (the outputs of that launch are then undefined). */
mlora_status mlora_sync_status(const mlora_plan_t* plan, void* stream);

/* Number of fp32 elements of H / dH: sum_i n_i r_i. */
int64_t mlora_h_elems(const mlora_plan_t* plan);

/* Inspect the plan's host tables (for tests and tooling).  `what` selects a
 * table (MLORA_Q_*); up to `cap` int64 values are copied to `out` and the
 * table's full length is stored in *count.  Tables:
 *   MLORA_Q_SUMMARY : N, d_in, d_out, n_segs, n_mtiles, C_total, n_chunks, n_images,
 *                     n_items(shrink), n_items(dA), n_items(dB), workspace_bytes
 *   MLORA_Q_MTILES  : per 128-row tile: first job, last job, first chunk, chunk count, image offset
 *   MLORA_Q_COLUMNS : per job: first column of its rank window, padded width
 *   MLORA_Q_WGRAD_A : per dA work item, CTA by CTA: row block, job, first and end half-tile, first
 *                     chunk, chunks, part, parts, CTA (an item whose tokens the schedule cuts
 *                     across CTAs runs as `parts` items; parts = 1 for a whole item)
 *   MLORA_Q_WGRAD_B : per dB work item: same fields
 *   MLORA_Q_WINDOW  : per single-CTA shrink / dH work item: tile, first chunk, chunks, first dH K
 *                     slice, dH K slices
 *   MLORA_Q_ADAPTERS: per segment-table entry: job, first packed column, rank, first and end
 *                     output column of its B
 *   MLORA_Q_WINDOW_PAIRS: 1 if the shrink / dH run on CTA pairs, else 0; then the CTA pairs'
 *                     work lists, pair by pair, one entry per item or piece: CTA pair, 256-token
 *                     pair of tiles, first chunk, chunks (even), first shrink K slice, shrink K
 *                     slices, first dH K slice, dH K slices, piece, pieces (an item the schedule
 *                     cuts along K runs as `pieces` entries on different pairs; 1 = whole item)
 *   MLORA_Q_GEMM_FWD / MLORA_Q_GEMM_BWD: the CTA-pair base GEMM's work list in launch order:
 *                     raster order (1 = groups of output tiles sweep the token pairs, 0 = groups
 *                     of token pairs sweep the output tiles), group size, items, full-width
 *                     items, CTA pairs launched; then per item: token pair, first output column,
 *                     width (256, or 128 for the halves of a split last wave) */
#define MLORA_Q_SUMMARY 0
#define MLORA_Q_MTILES 1
#define MLORA_Q_COLUMNS 2
#define MLORA_Q_WGRAD_A 3
#define MLORA_Q_WGRAD_B 4
#define MLORA_Q_WINDOW 5
#define MLORA_Q_ADAPTERS 6
#define MLORA_Q_WINDOW_PAIRS 7
#define MLORA_Q_GEMM_FWD 8
#define MLORA_Q_GEMM_BWD 9
mlora_status mlora_plan_describe(const mlora_plan_t* plan, int32_t what, int64_t* out, int64_t cap,
                                 int64_t* count);

/* Per-kernel timing, for tooling.  While enabled, every launch the plan makes is bracketed by
 * two CUDA events recorded on the launching stream (so the measured time is the kernels' own,
 * in stream order).  mlora_profile_read() waits for the recorded events, stores for each kernel
 * id the summed milliseconds (ms[id]) and the number of timed launches (launches[id]) for ids
 * below cap, sets *n_kernels to the number of ids, and clears the record.  Either array may be
 * NULL.  The plan is not thread-safe while profiling. */
mlora_status mlora_profile_enable(mlora_plan_t* plan, int32_t enable);
mlora_status mlora_profile_read(mlora_plan_t* plan, double* ms, int64_t* launches, int32_t cap,
                                int32_t* n_kernels);

/* Name of a kernel id of mlora_profile_read ("fwd_gemm", "adamw", ...; "" if out of range). */
const char* mlora_kernel_name(int32_t id);

/* Number of CUDA kernels this library has launched in this process so far. */
int64_t mlora_launch_count(void);

/* Device memory of one packed layer, in bytes (the single-GPU capacity check of the memory
 * model in "PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §8, for one
 * layer of one device).  lora_params is the paper's M_lora_param with fp32 masters (4 bytes
 * per parameter); lora_grad_state is c_grad = 3 times it (gradient, first and second moment:
 * the page multiplies by the precision a second time, which double-counts the bytes; read
 * as c_grad x M_lora_param); lora_act is the paper's M_lora_act (b x s x r per job = H, fp32)
 * plus the backward's dH of the same size.  The others are this library's buffers. */
typedef struct mlora_memory {
    int64_t base_weight;      /* W */
    int64_t activations;      /* X, Y, dY, dX */
    int64_t lora_params;      /* A_i, B_i */
    int64_t lora_grad_state;  /* dA_i, dB_i and the AdamW moments */
    int64_t lora_act;         /* H and dH */
    int64_t workspace;        /* mlora_plan's workspace_bytes */
    int64_t plan_tables;      /* the plan's own device tables */
    int64_t total;
} mlora_memory;

/* Fill *out for the plan (host only; valid for host-only plans too). */
mlora_status mlora_memory_estimate(const mlora_plan_t* plan, mlora_memory* out);

/* Cost model of one training step of a pack on one GPU: T(H, 1) of "PLoRA: Efficient Concurrent
 * LoRA Training for Large Language Models", §3.1-§3.2 (the planner's throughput objective divides
 * by the step time T of a packed job; the page measures T from a job's first iterations).  Here T
 * comes from a table of measured steps of this library (forward + backward + AdamW, inputs in
 * device memory), one point per measured pack:
 *   d_in, d_out  the layer's shape
 *   n_tokens     N of the measured pack
 *   lora_work    sum over its adapters of n_i r_i (d_in + w_i), w_i = the output width of B_i
 *   step_ms      its measured step time
 * A pack's algorithmic work is F = 4 N d_in d_out + 6 lora_work (the FLOP count of one step).
 * Among the points with the plan's (d_in, d_out), sorted by F, T is interpolated linearly in F
 * between the two points around the plan's F; below the smallest and above the largest point it
 * is F divided by that point's rate F / step_ms.  With no point of that shape it is F divided by
 * the rate of the point whose F is nearest (in ratio) to the plan's.  *step_ms receives T in
 * milliseconds, *basis (may be NULL) 0 for an interpolation, 1 for a same-shape extrapolation, 2
 * for another shape's rate.  bf16 and 4-bit-base plans; MLORA_ERR_UNSUPPORTED for fp32 plans,
 * MLORA_ERR_INVALID for an empty table or a point with step_ms <= 0.  Host only. */
typedef struct mlora_cost_point {
    int32_t d_in;
    int32_t d_out;
    int64_t n_tokens;
    double lora_work;
    double step_ms;
} mlora_cost_point;

mlora_status mlora_cost_estimate(const mlora_plan_t* plan, const mlora_cost_point* table, int32_t n_points,
                                 double* step_ms, int32_t* basis);

/* Split whole jobs across n_ranks GPUs that each hold a replica of W (the layer shards by job
 * with no collective: every job's gradients and optimizer step stay on its GPU).  Jobs are
 * assigned longest-first to the least-loaded rank, with a job's cost taken as its share of
 * the step's arithmetic, n_i (d_in d_out + 3 r_i (d_in + d_out)).  rank_of_job[i] receives the
 * rank of segs[i]; load[r] (may be NULL, n_ranks entries) the summed cost of rank r.  Host only. */
mlora_status mlora_shard_jobs(const mlora_problem* problem, const mlora_segment* segs, int32_t n_segs,
                              int32_t n_ranks, int32_t* rank_of_job, double* load);

/* mlora_shard_jobs for jobs that train one adapter on each of several projections with the same
 * tokens and rank (the projections of a decoder layer, each its own problem): a job's cost is
 * the sum over the n_problems projections of n_i (d_in d_out + 3 r_i (d_in + d_out)), and every
 * projection of a job goes to the same rank.  segs holds one entry per job (tok_offset,
 * n_tokens and rank are read; pointers are ignored).  mlora_shard_jobs is this call with one
 * problem.  Host only. */
mlora_status mlora_shard_jobs_multi(const mlora_problem* problems, int32_t n_problems, const mlora_segment* segs,
                                    int32_t n_segs, int32_t n_ranks, int32_t* rank_of_job, double* load);

/* Forward pass without a caller workspace, for callers that cannot allocate device memory
 * when they run the layer (a runtime that forbids cudaMalloc after start-up, a framework whose
 * memory comes only from its own pools, code running while another thread captures a graph).
 * The paper has no counterpart; this is a deployment convenience.
 *
 * Same arguments and results as mlora_forward, minus `workspace`: the scratch is one static
 * device array of 64 MiB that the library holds on every GPU it is loaded on until the
 * process exits.  This call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  Its first call on a device looks up that array's device address on the current
 * device (a one-time set-up per device).
 * Plans whose forward needs more scratch than 64 MiB, and plans with a 4-bit base
 * (MLORA_BF16_W4), are rejected with MLORA_ERR_UNSUPPORTED and a message in
 * mlora_last_error(); use mlora_forward / mlora_forward_w4 for them.  All calls on a device
 * share the one array and it keeps the last call's contents: because another plan may have
 * written it since, every call rebuilds the plan's bf16 adapter copies in it (MLORA_REUSE_STAGING
 * never skips that step here), so nothing in it needs to start at zero.  Calls that overlap on
 * the GPU (different streams without ordering between them) race on it, so order them on one
 * stream or with events. */
mlora_status mlora_forward_static_ws(const mlora_plan_t* plan, const void* X, const void* Wt, void* Y, float* H,
                                     void* stream);

/* Human-readable name of a status code (static storage). */
const char* mlora_status_string(mlora_status s);

/* Text of the last error raised on this host thread ("" if none). */
const char* mlora_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t mlora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
