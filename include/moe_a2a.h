/*
 * moe_a2a.h -- C ABI of the GB300-native top-k expert-parallel dispatch /
 * combine library (libmoe_a2a.so).
 *
 * The ep_size "ranks" are logical partitions of ONE GPU's memory: dispatch
 * scatters token rows into a padded receive workspace laid out per
 * destination rank, combine gathers each token's per-rank messages back and
 * reduces them once.  There is no peer memory, no NVLink traffic and no
 * collective.
 *
 * Sources of the operations (web pages, cited by title and section):
 *   [IX] SemiAnalysisAI/InferenceX PR #2450, "CollectiveX: add FlashInfer
 *        one-sided NVLink EP for the GB SKUs": "The adapter" table (phase
 *        contract; receive padded [ep_size, runtime_max_tokens_per_rank,
 *        hidden]; runtime_max_tokens_per_rank <= max_num_tokens, workspace
 *        sized once), the on-metal probe comment (the MoeAlltoAll
 *        __init__/dispatch/combine signatures), the bring-up run table
 *        (routing metadata as payloads, non-local expert ids masked,
 *        local_expert_counts), "Kernel arithmetic read from source"
 *        (fp32 accumulation, round-to-nearest-even bf16 store), "Best
 *        remaining lead" (recv counters are the authoritative per-source
 *        counts), "Update -- the correctness failures are resolved"
 *        (fp32 accumulator with a single narrowing; the combine payload can
 *        be written straight into the workspace).
 *   [VL] vllm-project/vllm PR #41382, "[Bugfix] Fix double reduce in
 *        flashinfer_nvlink_two_sided and flashinfer_nvlink_one_sided
 *        backends": the combine output is already reduced and is final.
 *   [MG] magik.net, "Fusing the Allreduce: A Precision Investigation into
 *        FlashInfer's Verify-Path Optimization", "The Message Itself": the
 *        reduction is fused with residual add + RMSNorm in one kernel.
 *
 * Notation: R = ep_size, M = max_tokens_per_rank, m = runtime max of one
 * call (T <= m <= M), T = tokens per source rank of one call, H = hidden,
 * E = num_experts, K = top_k, Epr = E / R.  Expert e lives on rank e / Epr.
 * bf16 tensors are IEEE bfloat16 bit patterns, row-major, dense.
 *
 * Ownership: the caller owns every device buffer, including the workspace.
 * The handle owns host state only.  Views returned by moe_dispatch alias the
 * workspace and stay valid until the next moe_dispatch on the handle.
 *
 * Errors: every entry point returns a moe_status code and never aborts.  A
 * call that returns an error leaves the phase unchanged.  Host-side checks
 * (sizes, pointers, alignment, phase) run before anything is queued.
 * Expert ids outside [-1, E) are detected on the device: the entry is
 * skipped and a sticky device flag is raised, which moe_a2a_get_error
 * reads.  Expert id -1 (the invalid_token_expert_id sentinel) means "no
 * expert" and is skipped silently.
 *
 * Streams: `stream` arguments are cudaStream_t values passed as void*
 * (NULL = the legacy default stream).  All work of a call is ordered on
 * that stream: moe_dispatch in the rank layout runs the second half of its
 * routing pass on a stream the handle creates at its first dispatch,
 * forked from `stream` by an event after the first half and joined back
 * into `stream` by another event before the call returns, so later work on
 * `stream` sees every output, and capturing `stream` into a CUDA graph
 * captures both branches.  Calls return without synchronising, except
 * moe_a2a_get_error.  A handle is bound to the CUDA device that is current
 * at its first dispatch; moe_a2a_destroy releases its stream and events.
 *
 * CUDA graphs: calls made while `stream` is capturing queue the same
 * kernels and memsets into the graph; a replay runs them with the pointers,
 * sizes and options of the capture, on whatever the buffers hold then (the
 * host-side phase is not replayed).  Every call's device state is cleared
 * inside the call, so captured dispatch / combine pairs can be replayed any
 * number of times (moe_dispatch takes its routing passes while capturing,
 * see below).
 *
 * Host threads: a handle keeps host-side state (phase, views, which count
 * buffer is current), so calls on one handle must not run concurrently;
 * distinct handles are independent.  Handles of different sizes may share
 * one process and device: a kernel's dynamic shared-memory limit, which is
 * one per process, is raised to the largest size a handle needs and never
 * lowered.
 *
 * Errors: MOE_ERR_CUDA means a CUDA call of the library failed; the
 * runtime's last error (cudaGetLastError) is cleared before returning, so
 * that it is not reported again by the caller's next CUDA call.
 */
#ifndef MOE_A2A_H
#define MOE_A2A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad config, NULL/misaligned pointer, bad size */
    MOE_ERR_PHASE = 2,         /* dispatch twice without combine, or combine
                                  without a dispatch ([IX] "The adapter") */
    MOE_ERR_CAPACITY = 3,      /* runtime_max > max_tokens_per_rank, or
                                  tokens_per_rank > runtime_max */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_ROUTING = 5,       /* device flag: an expert id outside [-1, E) */
    MOE_ERR_DEVICE_TIMEOUT = 6,/* device flag: a bounded on-chip wait ran out */
    MOE_ERR_INTERNAL = 7,      /* device flag: a consistency guard fired (a
                                  routing slot outside its plane was skipped);
                                  never expected, reported rather than faulting */
    MOE_ERR_SETUP_IN_CAPTURE = 8 /* moe_route_static_scratch: the first call in
                                  a CUDA context came while `stream` was
                                  capturing; nothing was queued */
};

/* Bits of the sticky device flag word (see moe_a2a_get_error). */
#define MOE_DEVICE_FLAG_BAD_EXPERT_ID 0x1u
#define MOE_DEVICE_FLAG_WAIT_TIMEOUT 0x2u
#define MOE_DEVICE_FLAG_BAD_SLOT 0x4u

/* Limits checked by moe_a2a_create. */
#define MOE_MAX_EP_SIZE 32
#define MOE_MAX_TOP_K 32
#define MOE_MAX_EXPERTS 8192
#define MOE_MAX_HIDDEN 16384

/* Sizes fixed for the life of a handle ([IX] MoeAlltoAll __init__:
 * max_num_tokens, top_k, num_experts, hidden_size; the workspace is sized
 * once from max_tokens_per_rank). */
typedef struct moe_a2a_config {
    int32_t ep_size;             /* R, 1..32 logical ranks */
    int32_t max_tokens_per_rank; /* M >= 1 */
    int32_t hidden;              /* H, multiple of 8, 8..16384 */
    int32_t num_experts;         /* E, multiple of R, <= 8192 */
    int32_t top_k;               /* K, 1..32 */
} moe_a2a_config_t;

typedef struct moe_a2a moe_a2a_t;

/* Device pointers into the workspace, produced by moe_dispatch.  All arrays
 * are dense with plane stride m = runtime max of the call ([IX] "The
 * adapter": padded, not compact).  Slots j >= recv_counts[d][s] of a plane
 * are padding: never written by dispatch and never read by combine. */
typedef struct moe_dispatch_view {
    void *recv_x;                 /* bf16  [R dst][R src][m][H] */
    int32_t *recv_topk_ids;       /* int32 [R][R][m][K]: expert id if it lives
                                     on dst, else -1 (non-local masking) */
    float *recv_topk_w;           /* fp32  [R][R][m][K]: weight if local, else 0 */
    int32_t *src_token;           /* int32 [R][R][m]: source token of slot j */
    int32_t *recv_counts;         /* int32 [R dst][R src] */
    int32_t *local_expert_counts; /* int32 [R][Epr]: valid (token, k) entries
                                     per local expert, over all sources (one of
                                     two workspace regions: take the pointer
                                     from each call's view) */
    int32_t *send_slot;           /* int32 [R src][T][send_stride]: slot of
                                     token (s,t) in plane (d,s), -1 if not sent */
    float *dest_weight;           /* fp32 [R src][T][send_stride]: sum, in
                                     ascending k, of the token's top-k weights
                                     whose expert lives on d (0 if not sent) */
    int32_t plane_stride;         /* m */
    int32_t tokens_per_rank;      /* T (moe_dispatch), -1 (moe_dispatch_varlen) */
    int32_t send_stride;          /* R rounded up to a multiple of 4 */
    int32_t token_stride;         /* rows per source rank of the token arrays
                                     (x, send_slot, dest_weight, residual, out):
                                     T, or m for moe_dispatch_varlen */
    float *recv_scale;            /* fp32 per-row scale of recv_x in the FP8
                                     receive format ([R][R][m], or [E][cap]
                                     in the expert layout), else NULL */
    int32_t recv_format;          /* MOE_FORMAT_* of recv_x */
    int32_t layout;               /* MOE_LAYOUT_* of the handle */
    int32_t kernels;              /* kernels this dispatch queued (0 for an
                                     empty call: memsets only) */
} moe_dispatch_view_t;

/* Bytes of device workspace a handle with this config needs (0 if the
 * config is invalid).  Sized once for max_tokens_per_rank ([IX] "The
 * adapter": workspace sized once from the ladder maximum). */
size_t moe_a2a_workspace_bytes(const moe_a2a_config_t *cfg);

/* ---- Receive layouts --------------------------------------------------------
 * MOE_LAYOUT_RANK (moe_a2a_create): one plane per (destination rank, source
 *   rank), one row per (token, destination rank), as described above.
 * MOE_LAYOUT_EXPERT (moe_a2a_create_layout): every received row carries a
 *   single expert -- [IX] the association-order analysis ("the low-latency
 *   padded layouts", whose rows carry one expert each) and the harness
 *   review ("weighted-kernel-sum": the combine kernel applies the gates).
 *   Readings: expert e has a plane of cap = R * m rows (R * M in the
 *   workspace); one row per distinct (token, expert) whose id is valid and
 *   whose rank is active, rows in ascending (source rank, token).  The view
 *   of a dispatch then holds
 *     recv_x       bf16 [E][cap][H] (e4m3 [E][cap][H] in the FP8 format)
 *     recv_topk_w  fp32 [E][cap]: the row's weight wsum (below)
 *     recv_topk_ids NULL (a row's expert is its plane)
 *     src_token    int32 [E][cap]: s * token_stride + t of the row's token
 *     recv_counts  int32 [E]: rows per expert
 *     local_expert_counts int32 [E]: valid (token, k) entries, duplicates
 *                  included
 *     send_slot    int32 [R][token_stride][send_stride]: entry k = the
 *                  absolute row e_k * cap + slot of recv_x for the first k
 *                  carrying that expert; -1 for later duplicates, absent or
 *                  dead experts and entries k >= K
 *     dest_weight  fp32, same shape: wsum = sum over the token's slots with
 *                  that expert, ascending k, of its weights from +0.0 (0
 *                  where send_slot is -1)
 *     plane_stride cap; send_stride = top_k rounded up to a multiple of 4.
 *   Combine sums, per token, over k ascending with send_slot >= 0, of
 *   v = expert_out[row] (weighted = 0) or wsum * v (weighted = 1) in fp32
 *   from +0.0, no FMA, then the epilogue of moe_combine; expert_out is
 *   [E][cap][H].  Requires num_experts <= 1024; the bf16 top-k tree
 *   reduction is not available in this layout.  The workspace grows as
 *   E * R * M * H (two bf16 regions): this layout is meant for decode-sized
 *   batches. */
enum moe_layout { MOE_LAYOUT_RANK = 0, MOE_LAYOUT_EXPERT = 1 };

/* Expert-side consumer of the expert planes ([IX] "Why": between dispatch
 * and combine each expert applies its own weights to the rows it received;
 * vLLM applies the gates in the MoE layer around it).  Reading: one linear
 * map per expert, W_e of N x H stored as a linear layer stores it (row n =
 * the weights of output n).  For every expert e and received row
 * j < recv_counts[e] of the current dispatch:
 *   out[e][j][n] = bf16_rn( sum_h x[e][j][h] * w[e][n][h] ),
 * bf16 products accumulated in fp32 on the tensor cores (tcgen05; the order
 * of the additions is the hardware's).  Rows past a count are not written.
 *   d_w   bf16 [E][N][H], 16-byte aligned;
 *   N     a multiple of 128; the hidden size H must be a multiple of 64;
 *   d_out bf16 [E][cap][N] (cap = plane_stride of the dispatch), or NULL to
 *         write the combine payload region (then N must equal H), so that
 *         moe_combine(h, NULL, ...) reduces the experts' outputs.
 * Requires the expert layout and the bf16 receive format, and a pending
 * dispatch (MOE_ERR_PHASE otherwise); the phase does not change.  Queues one
 * kernel on `stream`. */
int moe_expert_gemm(moe_a2a_t *h, const void *d_w, int32_t N, void *d_out, void *stream);

/* The same product on FP8 operands (tcgen05 .kind::f8f6f4, e4m3 x e4m3 into
 * fp32), for a dispatch made in the FP8 receive format: the rows are the
 * e4m3 codes qx with their per-row scales sx (recv_scale), the weights e4m3
 * codes qw [E][N][H] with one fp32 scale per output channel sw [E][N]
 * (reading: dequantised operands, the FP8 payload of [IX] "The adapter"):
 *   out[e][j][n] = bf16_rn( (sum_h f(qx) * f(qw)) * sx[e][j] * sw[e][n] ),
 * the products of e4m3 values exact, the sum in fp32 on the tensor cores,
 * then two fp32 multiplies.  H must be a multiple of 128, N of 128; d_w8
 * 16-byte and d_w_scale 4-byte aligned; d_out as for moe_expert_gemm (bf16,
 * NULL = the combine payload when N == H).  Requires the expert layout and
 * the FP8 receive format. */
int moe_expert_gemm_fp8(moe_a2a_t *h, const void *d_w8, const float *d_w_scale, int32_t N,
                        void *d_out, void *stream);

/* The expert-side product on the rank planes that moe_dispatch produces in
 * the rank layout ([IX] "Why": each expert applies its weights to the rows
 * it received; vLLM applies the gates in the MoE layer).  A received row
 * (d, s, j), j < recv_counts[d][s], carries one token and, in recv_topk_ids,
 * the token's experts that live on rank d.  For every such row and column n:
 *   y_k[n]  = bf16_rn( sum_h x[d][s][j][h] * w[e_k][n][h] )   (e_k local;
 *             bf16 products accumulated in fp32 on the tensor cores),
 *   out[d][s][j][n] = bf16_rn( sum over k ascending with a local e_k of
 *             g_k * y_k[n] ),  g_k = recv_topk_w[d][s][j][k] if apply_gates
 *             else 1, in fp32 from +0.0, one multiply and one add per term.
 * With apply_gates and out = the combine payload, an unweighted
 * moe_combine(h, NULL, 0, ...) then returns sum_k w_k * y_k per token.
 *   d_w      bf16 [E][N][H] (row n = the weights of output n), 16-byte aligned;
 *   N        a multiple of 128; H must be a multiple of 64; E <= 1024;
 *   d_out    bf16 [R][R][m][N], or NULL for the combine payload (N == H);
 *            rows past a plane's count are not written;
 *   d_scratch caller-owned device memory of at least
 *            moe_expert_gemm_rank_scratch_bytes(cfg, N) bytes, 256-byte
 *            aligned (pair lists and the experts' bf16 outputs; contents
 *            need not be initialised, and are garbage afterwards).
 * Requires the rank layout and the bf16 receive format (MOE_ERR_INVALID_ARG
 * otherwise), R * R * m < 2^31, a pending dispatch (MOE_ERR_PHASE); the
 * phase does not change.
 * MOE_ERR_CAPACITY if scratch_bytes is too small.  Queues a memset and three
 * kernels on `stream` (pair lists, the gathered tcgen05 product, the gated
 * sum per row). */
size_t moe_expert_gemm_rank_scratch_bytes(const moe_a2a_config_t *cfg, int32_t N);

int moe_expert_gemm_rank(moe_a2a_t *h, const void *d_w, int32_t N, int32_t apply_gates,
                         void *d_out, void *d_scratch, size_t scratch_bytes, void *stream);

/* moe_expert_gemm_rank on FP8 operands (tcgen05 .kind::f8f6f4, e4m3 x e4m3
 * into fp32), for a rank-layout dispatch made in the FP8 receive format: the
 * rows are the e4m3 codes qx with one scale sx per received row (the
 * dispatch's recv_scale [R][R][m]), the weights e4m3 codes qw [E][N][H] with
 * one fp32 scale per output channel sw [E][N] (reading: dequantised
 * operands, the FP8 payload of [IX] "The adapter", as moe_expert_gemm_fp8):
 *   y_k[n]  = bf16_rn( (sum_h f(qx[h]) * f(qw[e_k][n][h])) * sx * sw[e_k][n] ),
 * the products of e4m3 values exact, the sum in fp32 on the tensor cores,
 * then two fp32 multiplies; the message is the gated sum of
 * moe_expert_gemm_rank, in fp32 from +0.0 in ascending k, narrowed once.
 * H must be a multiple of 128, N of 128, E <= 1024; d_w8 16-byte and
 * d_w_scale 4-byte aligned; d_out, d_scratch (the same size:
 * moe_expert_gemm_rank_scratch_bytes) and the errors as for
 * moe_expert_gemm_rank, with the FP8 receive format required.  Queues a
 * memset and three kernels on `stream`. */
int moe_expert_gemm_rank_fp8(moe_a2a_t *h, const void *d_w8, const float *d_w_scale, int32_t N,
                             int32_t apply_gates, void *d_out, void *d_scratch,
                             size_t scratch_bytes, void *stream);

/* moe_a2a_workspace_bytes for a layout (0 if the pair is invalid). */
size_t moe_a2a_workspace_bytes_layout(const moe_a2a_config_t *cfg, int32_t layout);

/* Create a handle over a caller-owned device workspace of at least
 * moe_a2a_workspace_bytes(cfg) bytes, 256-byte aligned.  Host-only: queues
 * nothing and needs no GPU.  On success *out receives the handle in the
 * IDLE phase. */
int moe_a2a_create(const moe_a2a_config_t *cfg, void *d_workspace,
                   size_t workspace_bytes, moe_a2a_t **out);

/* moe_a2a_create for a layout (MOE_LAYOUT_*); the layout is fixed for the
 * life of the handle.  MOE_ERR_INVALID_ARG for an unknown layout or a config
 * the layout cannot take. */
int moe_a2a_create_layout(const moe_a2a_config_t *cfg, int32_t layout, void *d_workspace,
                          size_t workspace_bytes, moe_a2a_t **out);

/* Dispatch ([IX] dispatch(token_selected_experts, input_payloads,
 * runtime_max_tokens_per_rank, invalid_token_expert_id)).
 *   d_topk_ids  int32 [R][T][K], 4-byte aligned; -1 = no expert
 *   d_topk_w    fp32  [R][T][K], 4-byte aligned
 *   d_x         bf16  [R][T][H], 16-byte aligned
 *   tokens_per_rank T (0 <= T <= runtime_max), runtime_max m (1 <= m <= M).
 * Routes every token to each distinct rank owning one of its experts (one
 * message per (token, rank)), assigns slots in ascending source-token order
 * within each (destination, source) plane, copies x rows and the masked
 * top-k metadata into the planes, and counts rows per plane and per local
 * expert.  Queues one kernel on `stream` when every source holds the same
 * number of tokens, at most 256 (bf16 rows, either layout; FP8 rows: 128 in
 * the rank layout, 64 in the expert layout), and `stream`
 * is not capturing into a CUDA graph (that kernel alternates two count
 * buffers between calls, which a replay cannot follow; in the expert layout
 * the rows per expert alternate with them, so read them through the view);
 * else three (the rank layout's second on the handle's own stream, as
 * described above).  IDLE -> DISPATCHED; returns
 * MOE_ERR_PHASE if already DISPATCHED.  If out_view is not NULL it receives
 * the views of this call. */
int moe_dispatch(moe_a2a_t *h, const int32_t *d_topk_ids, const float *d_topk_w,
                 const void *d_x, int32_t tokens_per_rank,
                 int32_t runtime_max_tokens_per_rank, void *stream,
                 moe_dispatch_view_t *out_view);

/* Dispatch with a token count per source rank (the pages' upstream API
 * sizes each rank's batch separately; the readings: tokens past a rank's
 * count are absent, exactly as if their expert ids were all -1, and nothing
 * of theirs is read or written).
 *   tokens_per_rank: HOST array of R counts, each 0..runtime_max.
 *   d_topk_ids int32 [R][m][K], d_topk_w fp32 [R][m][K], d_x bf16 [R][m][H]:
 *   the rows of source s are s*m + t for t < tokens_per_rank[s]; the rows
 *   past a count are never read.
 * Everything else as moe_dispatch; the following moe_combine reads residual
 * and writes out / residual_out with the same [R][m][H] row layout and
 * leaves the rows past each count untouched. */
int moe_dispatch_varlen(moe_a2a_t *h, const int32_t *d_topk_ids, const float *d_topk_w,
                        const void *d_x, const int32_t *tokens_per_rank,
                        int32_t runtime_max_tokens_per_rank, void *stream,
                        moe_dispatch_view_t *out_view);

/* Mark which logical ranks take part ([IX] upstream combine's
 * active_rank_mask; "dead-rank" marking).  Bit d set = rank d is alive.
 * Dispatch treats an expert that lives on a dead rank exactly as an absent
 * expert (id -1): no message, not counted, masked in the metadata rows;
 * combine skips the messages of ranks that are dead at combine time (also
 * those sent before the rank was marked dead).  Default: all ranks alive.
 * Host-only; returns MOE_ERR_INVALID_ARG for bits at or above ep_size. */
int moe_a2a_set_active_ranks(moe_a2a_t *h, uint32_t active);

/* Device pointer to the combine payload region of the workspace ([IX]
 * get_combine_payload_tensor_in_workspace): bf16 [R][R][m][H] with the m of
 * the current dispatch.  Experts may write their outputs here and pass
 * NULL (or this pointer) as d_expert_out, so combine needs no staging copy.
 * NULL if h is NULL. */
void *moe_combine_payload(moe_a2a_t *h);

/* Combine ([IX] combine(payload, runtime_max_tokens_per_rank,
 * payload_in_workspace); [VL]; [MG]).  For each source token (s,t):
 *   acc = sum over its destination ranks d, ascending d, of
 *         v = expert_out[d][s][send_slot(s,t,d)][:]  (weighted = 0), or
 *         dest_weight(s,t,d) * v                      (weighted != 0),
 *   in fp32 starting from +0.0, one IEEE multiply and one add per term
 *   (no FMA); each message is read exactly once and the result is final
 *   (it must not be reduced again).
 * Unfused (d_residual == NULL): d_out[s][t][:] = bf16_rn(acc).
 * Fused: hsum = acc + residual (fp32); d_residual_out = bf16_rn(hsum) if
 *   not NULL (it may be the same buffer as d_residual);
 *   d_out = bf16_rn(hsum * rsqrt(mean(hsum^2) + eps) * gamma).
 *   d_expert_out bf16 [R][R][m][H] (NULL = the in-workspace payload region;
 *       the recv_x view is also accepted, i.e. identity experts)
 *   d_residual, d_residual_out, d_out bf16 [R][T][H]; d_gamma bf16 [H]
 *   All bf16 pointers 16-byte aligned.  d_out must not overlap any input.
 * Queues one kernel on `stream`.  DISPATCHED -> IDLE; returns MOE_ERR_PHASE
 * if no dispatch is pending. */
int moe_combine(moe_a2a_t *h, const void *d_expert_out, int32_t weighted,
                const void *d_residual, const void *d_gamma, float eps,
                void *d_out, void *d_residual_out, void *stream);

/* Synchronise `stream`, read and clear the sticky device flag word.
 * Returns MOE_OK if no flag was set, MOE_ERR_ROUTING if an expert id outside
 * [-1, E) was seen, MOE_ERR_DEVICE_TIMEOUT if a bounded wait ran out (the
 * kernel then stopped early and its outputs are incomplete), or
 * MOE_ERR_CUDA.  If flags is not NULL it receives the raw bits. */
int moe_a2a_get_error(moe_a2a_t *h, void *stream, uint32_t *flags);

/* Free the handle (host memory only; the workspace stays the caller's). */
int moe_a2a_destroy(moe_a2a_t *h);

/* Phase of the handle: 0 = IDLE, 1 = DISPATCHED, -1 if h is NULL. */
int moe_a2a_phase(const moe_a2a_t *h);

/* Static text for a status code. */
const char *moe_a2a_status_string(int status);

/* Reduction used by moe_combine.
 * MOE_REDUCE_FP32_RANK_ORDER (default): fp32 sum over destination ranks in
 *   ascending order, one narrowing ([IX] "Update": the fp32 accumulator of
 *   version 0.6.16 on, "domain-fp32").
 * MOE_REDUCE_BF16_TOPK_TREE (rank layout only): the reduction of FlashInfer's one-sided combine
 *   through version 0.6.15 ([IX] "Update", "topk-slot-tree"): one bf16
 *   accumulator per top-k slot, each rank's message in the first slot whose
 *   expert lives on that rank (later slots of the same rank and invalid ids
 *   hold zero), reduced by the pairwise tree (a0+a1)(a2+a3)...; (a0+a2)...;
 *   (a0+a4) with a bf16 rounding after every add (slots padded with zeros to
 *   a power of two).  Unweighted only (moe_combine with weighted != 0
 *   returns MOE_ERR_INVALID_ARG); requires top_k <= 8.  The fused epilogue,
 *   when requested, applies to the tree's result. */
enum moe_reduction { MOE_REDUCE_FP32_RANK_ORDER = 0, MOE_REDUCE_BF16_TOPK_TREE = 1 };

/* Select the reduction of subsequent moe_combine calls (host-only).
 * Returns MOE_ERR_INVALID_ARG for an unknown mode or top_k > 8 with the tree. */
int moe_a2a_set_reduction(moe_a2a_t *h, int32_t reduction);

/* ---- FP8 payloads ----------------------------------------------------------
 * [IX] "The adapter" (the paragraph on why the adapter is BF16-only): an FP8
 * dispatch carries a scale payload beside the rows and is validated against
 * the cast round trip; the upstream combine can emit FP8 outputs ([IX] the
 * comment on the shipped combine signature: upstream output_dtype /
 * use_low_precision).  Readings: OCP FP8 E4M3 (bias 7, largest finite 448,
 * no infinities), one scale per token row:
 *   scale = amax_h |v_h| / 448 in binary32 (1 for an all-zero row),
 *   q_h   = e4m3(v_h / scale), binary32 division, round-to-nearest-even,
 *           magnitudes past 448 saturate to 448, NaN stays NaN;
 * dequantised value q_h * scale.
 *
 * Receive format (host-only, IDLE phase only; MOE_ERR_PHASE otherwise):
 *   MOE_FORMAT_BF16 (default): recv_x bf16 [R][R][m][H], recv_scale NULL.
 *   MOE_FORMAT_FP8_E4M3: dispatch writes recv_x as e4m3 bytes [R][R][m][H]
 *     (the first half of the bf16 region) with v = the bf16 row x[s][t], and
 *     recv_scale fp32 [R][R][m]; the metadata rows, counts and send tables
 *     are unchanged.  Needs H a multiple of 16 (MOE_ERR_INVALID_ARG).
 *   The expert outputs that combine reads stay bf16 in either format. */
enum moe_format { MOE_FORMAT_BF16 = 0, MOE_FORMAT_FP8_E4M3 = 1 };

int moe_a2a_set_recv_format(moe_a2a_t *h, int32_t format);

/* Combine with an FP8 output: the reduction and the fused epilogue exactly as
 * moe_combine (fp32 rank-order reduction only: MOE_ERR_INVALID_ARG with the
 * bf16 top-k tree), then, per token row, v = the fp32 result that moe_combine
 * would narrow to bf16 (acc unfused; the RMSNorm output fused) is quantised
 * as above into
 *   d_out_fp8   e4m3 [R][T][H] (16-byte aligned) and
 *   d_out_scale fp32 [R][T]    (4-byte aligned).
 * d_residual_out stays bf16.  Queues one kernel; DISPATCHED -> IDLE. */
int moe_combine_fp8(moe_a2a_t *h, const void *d_expert_out, int32_t weighted,
                    const void *d_residual, const void *d_gamma, float eps,
                    void *d_out_fp8, float *d_out_scale, void *d_residual_out,
                    void *stream);

/* The same per-row quantisation as a standalone call, for fp32 rows (e.g.
 * activations headed for an FP8 expert GEMM, or a check of the cast):
 *   d_x     fp32 [rows][H], 16-byte aligned, H a multiple of 8 (8..16384)
 *   d_q     e4m3 [rows][H], 16-byte aligned
 *   d_scale fp32 [rows], 4-byte aligned
 * rows >= 0 (0 queues nothing).  Queues one kernel on `stream`; no handle.
 * The quotients are the correctly rounded binary32 x / scale (one
 * reciprocal per row refined by FMA remainder steps, exact by Markstein's
 * theorem; rows with a scale outside [2^-100, 2^100] refine the pair
 * scaled by 2^100 or 2^-100, which leaves the quotient unchanged). */
int moe_quantize_rows_fp8(const float *d_x, int64_t rows, int32_t hidden, void *d_q,
                          float *d_scale, void *stream);

/* ---- Routing without any device allocation --------------------------------
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory: a plugin or custom op running
 * inside a framework that owns the whole device memory pool and exposes no
 * allocator, or a serving loop that forbids cudaMalloc after start-up
 * (cudaMalloc can synchronise the device and fragments a fixed budget).
 *
 * It runs the same routing pass as moe_dispatch (destination dedup,
 * ascending-token slots, send table, per-destination weights, source map,
 * masked metadata rows, recv counts, local-expert counts) into buffers the
 * caller passes, and keeps the pass's temporary memory in a file-scope
 * device array of MOE_STATIC_SCRATCH_BYTES.  The library allocates nothing
 * (no cudaMalloc/cudaFree, no allocating library call); the array is created
 * by the CUDA runtime on every device that loads the library and is held
 * until the process exits.
 *
 * Set-up: the first call in a CUDA context (with its device current) looks
 * up the array's device address with cudaGetSymbolAddress and keeps it with
 * the context's unique id; a later call in another context of that device
 * (after cudaDeviceReset, or after a framework recreated the primary
 * context, which reloads the library's device code) looks it up again, so a
 * stale address is never used.  Make the first call in each context before
 * any stream capture: a first call made while `stream` is capturing queues
 * nothing and returns MOE_ERR_SETUP_IN_CAPTURE.  All calls on a device share
 * the one array and it keeps the last
 * call's contents: calls whose work overlaps on the GPU (other streams, or
 * other threads without ordering) race on it and must be serialised by the
 * caller.  The parts that must start at zero (a ticket and an expert
 * histogram accumulator per source rank) are cleared at the start of every call
 * with cudaMemsetAsync on `stream`; the rest is written before it is read.
 *
 * Limit: moe_route_static_scratch_bytes(R, E, T) must not exceed
 * MOE_STATIC_SCRATCH_BYTES (2*R*ceil(T/256)*RP*4 + (R + R*E)*4 plus
 * alignment; e.g. R=8, E=256: up to T = 2092800) else MOE_ERR_CAPACITY.
 * Outputs (layouts as in moe_dispatch_view_t, RP = R rounded up to 4, all
 * 16-byte aligned): d_send_slot int32 [R][T][RP], d_dest_weight fp32
 * [R][T][RP], d_src_token int32 [R][R][m], d_recv_counts int32 [R][R],
 * d_local_expert_counts int32 [E], d_recv_topk_ids int32 [R][R][m][K],
 * d_recv_topk_w fp32 [R][R][m][K]; only valid slots of the [R][R][m]
 * arrays are written.  d_flags (optional, caller-zeroed uint32) receives
 * MOE_DEVICE_FLAG_BAD_EXPERT_ID if an id outside [-1, E) is seen.
 * Inputs: d_topk_ids int32 / d_topk_w fp32 [R][T][K], 4-byte aligned.
 * Queues two kernels on `stream`; no handle, no phase. */
#define MOE_STATIC_SCRATCH_BYTES (4u << 20)

size_t moe_route_static_scratch_bytes(int32_t ep_size, int32_t num_experts,
                                      int32_t tokens_per_rank);

int moe_route_static_scratch(int32_t ep_size, int32_t num_experts, int32_t top_k,
                             int32_t tokens_per_rank,
                             int32_t runtime_max_tokens_per_rank,
                             const int32_t *d_topk_ids, const float *d_topk_w,
                             int32_t *d_send_slot, float *d_dest_weight,
                             int32_t *d_src_token, int32_t *d_recv_counts,
                             int32_t *d_local_expert_counts,
                             int32_t *d_recv_topk_ids, float *d_recv_topk_w,
                             uint32_t *d_flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_A2A_H */
