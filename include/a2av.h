/*
 * a2av.h -- C ABI of a device-resident MoE dispatch/combine data plane for
 * GB300 (sm_103a): the data path of an AllToAllv whose split counts never
 * leave GPU memory.
 *
 * What the operation is.  NCCLX, "Collective Communication for 100k+ GPUs"
 * (Meta), Section 6.1, as told on the pages
 *   abhik.ai/papers/ncclx, section "Inference: small messages, unknown sizes";
 *   hungchun0201 research digest, section 3.3 "AllToAllvDynamic";
 *   qiguanping.github.io deep dive, section 7 (Figures 13, 16, 17):
 * a router picks the experts of each token, the tokens are sorted by expert
 * into a send buffer and an AllToAllv sends each one to the rank that holds
 * its expert (Figure 13); the counts live in GPU memory, are read when the
 * collective runs, only real tokens are sent (no padding to the worst case),
 * and the collective returns the counts it received; afterwards the expert
 * outputs come back and are combined.
 *
 * Here the R ranks are R windows in one GPU's memory, and the exchange is a
 * direct store of each token row into its destination window (no
 * intermediate send buffer).  Readings of what the pages leave open:
 *   - expert e lives on rank e / (E/R) (contiguous blocks);
 *   - "sorted by expert" is stable: expert, then token t, then slot j;
 *   - window d holds the segments of sources 0..R-1 back to back, in source
 *     order, with no gaps (the AllToAllv convention); or, in the
 *     expert-grouped receive order, the rows of local expert 0 from every
 *     source, then those of local expert 1, ... -- the layout one GEMM per
 *     local expert reads after the exchange (Inference section, Figure 13:
 *     the received tokens go on to their experts), the counts unchanged;
 *   - combine: out = bf16_rne(sum_j w_j * y[slot(t,j)]) accumulated in fp32
 *     from 0 in slot order, product and sum each rounded on its own.
 *
 * Conventions for every call below.
 *   - Every tensor pointer is a DEVICE pointer into memory of the plan's
 *     device, owned by the caller, row-major (C order), and must stay valid
 *     until the work enqueued on `stream` has finished.  The library never
 *     frees or retains them.
 *   - Row buffers (x, recv, y, out) must be 16-byte aligned and H % 8 == 0
 *     (rows move as 16-byte vectors); integer/float arrays 4-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Enqueueing calls are asynchronous: they return after
 *     launching and never synchronise, allocate, or read device memory back.
 *     Those that take a plan can be captured into a CUDA graph (the plan is
 *     made outside capture).  A returned A2AV_OK means "enqueued".
 *   - Host-side argument errors are returned synchronously
 *     (A2AV_ERR_INVALID_ARG) and nothing is enqueued.  Data errors found on
 *     the device (expert id out of range, fixed window too small) set sticky
 *     bits in the plan's device status word (A2AV_DEV_*), skip the offending
 *     store and never write out of bounds; read them with
 *     a2av_read_device_status outside capture.
 *   - A plan's workspace is shared by its calls: use one plan from one
 *     stream at a time (or order the streams).  Calls that overlap on the
 *     device through one plan race.
 *   - Stream order holds for every input: a call's kernels may become
 *     resident before the kernel ahead of them on the stream has finished
 *     (programmatic dependent launch), but none reads a tensor that kernel
 *     may write before it has completed.  So one call's `out` may be the next
 *     call's `x`, on the same stream, with nothing in between.  The pack and
 *     combine grids fill every SM: other work on the GPU during a call makes
 *     it slower, not wrong.
 *
 * Layouts (int32 unless said otherwise; R ranks, E experts, T tokens per
 * rank, H hidden, k experts per token, Epr = E/R):
 *   x            bf16  [R][T][H]           token rows, per source rank
 *   topk_idx     int32 [R][T][k]           global expert ids
 *   gate_w       fp32  [R][T][k]           combine weights
 *   recv, y      bf16  [arena_rows][H]     windows (recv layout)
 *   slot_map     int32 [R][T][k]           arena row of each assignment, -1 if dropped
 *   out          bf16  [R][T][H]
 *   splits.send_counts        [R][E]       rows rank s sends to expert e
 *   splits.send_offsets       [R][E]       exclusive scan of send_counts over e
 *   splits.recv_counts        [R][R]       [d][s] rows window d receives from s
 *   splits.recv_offsets       [R][R]       [d][s] exclusive scan over s
 *   splits.recv_expert_counts [R][R][Epr]  [d][s][le] = send_counts[s][d*Epr+le]
 *   splits.recv_expert_offsets [R][R][Epr] [d][s][le] window-relative first row of the
 *                                          rows s sends to local expert le of rank d:
 *                                          source order: recv_offsets[d][s] + s's rows for
 *                                          the lower local experts; expert order: all rows
 *                                          of the lower local experts + those of le from
 *                                          sources below s
 *   splits.recv_total         [R]          rows window d receives
 *   splits.window_base        [R]          arena row where window d starts
 */
#ifndef A2AV_H
#define A2AV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct a2av_plan_s *a2av_plan_t;

/* Host-side result of every call. */
typedef enum {
    A2AV_OK = 0,
    A2AV_ERR_INVALID_ARG = 1, /* bad config, null/misaligned pointer, size limit */
    A2AV_ERR_CUDA = 2,        /* a CUDA runtime call failed (message: a2av_last_error) */
    A2AV_ERR_NO_MEMORY = 3,   /* workspace allocation failed */
} a2av_status_t;

/* Sticky bits of the device status word. */
enum {
    A2AV_DEV_BAD_EXPERT = 1u << 0,      /* an expert id outside [0, E): dropped, slot -1 */
    A2AV_DEV_WINDOW_OVERFLOW = 1u << 1, /* fixed mode: a window got more than window_rows rows */
    A2AV_DEV_BAD_SLOT = 1u << 2,        /* combine/expert stand-in: a slot_map entry past the arena, skipped */
    A2AV_DEV_WAIT_TIMEOUT = 1u << 31,   /* a bounded wait on the kernel's own copies gave up (not expected) */
};

/* Window placement of the R destination windows in the recv arena. */
enum {
    A2AV_WINDOW_PACKED = 0, /* window d starts right after window d-1: arena of exactly R*T*k rows */
    A2AV_WINDOW_FIXED = 1,  /* window d owns rows [d*window_rows, (d+1)*window_rows) */
    A2AV_WINDOW_PADDED = 2, /* worst-case layout of a host-side AllToAllv under graph capture: every
                               (source s, destination d) pair owns T*k rows at (d*R + s)*T*k; the
                               padded baseline the dynamic collective is compared with */
};

/* Order of the rows inside each window (a2av_config_t.recv_order). */
enum {
    A2AV_ORDER_SOURCE = 0, /* AllToAllv convention: source segments in source order, each sorted by expert */
    A2AV_ORDER_EXPERT = 1, /* expert-grouped: local expert blocks in expert order, each holding its sources'
                              rows in source order; not with A2AV_WINDOW_PADDED */
};

/* Variant flags (a2av_config_t.flags). */
enum {
    A2AV_FLAG_PACK_LSU = 1u << 0,     /* pack+exchange with 16-byte vector loads/stores instead of TMA bulk copies */
    A2AV_FLAG_SPLITS_TILED = 1u << 1, /* always use the multi-CTA tiled splits kernel (else one CTA when it fits) */
    A2AV_FLAG_COMBINE_TMA = 1u << 2,  /* combine through TMA bulk copies into shared memory (default: vector gathers) */
    A2AV_FLAG_ROUTE_FUSED = 1u << 3,  /* a2av_route_splits: the router inside the tiled histogram kernel (default: the
                                         router kernel, then the splits kernel -- measured faster, see the call) */
    A2AV_FLAG_ROUTE_WARP = 1u << 4,   /* a2av_route: one warp per token on every shape (default: one lane per token
                                         where E % 4 == 0, k <= 8 and the logits are 16-byte aligned; same results) */
};

typedef struct {
    int32_t num_ranks;       /* R >= 1, <= 64 */
    int32_t num_experts;     /* E, a multiple of R, <= 2048 */
    int32_t tokens_per_rank; /* T >= 1; R*T*k < 2^31 */
    int32_t hidden;          /* H, a multiple of 8, >= 8 */
    int32_t topk;            /* k, 1..32 */
    int32_t window_mode;     /* A2AV_WINDOW_PACKED, A2AV_WINDOW_FIXED or A2AV_WINDOW_PADDED */
    int64_t window_rows;     /* fixed mode: rows per window (R*window_rows < 2^31); ignored when packed */
    int32_t device;          /* CUDA device ordinal the plan and all its tensors live on */
    uint32_t flags;          /* A2AV_FLAG_* */
    int32_t pack_ctas_per_sm; /* TMA pack: resident CTAs per SM, 1..4 (0 = 4) */
    int32_t pack_stage_bytes; /* TMA pack: bytes per shared-memory stage, multiple of 16
                                 (0 = 2 KiB for k >= 4, else min(row, 16 KiB)) */
    int32_t pack_store_lag;   /* TMA pack: row stores that may still read a stage before its refill, 1..8
                                 (0 = 6 for k >= 4, else 2) */
    int32_t combine_ctas_per_sm;  /* TMA combine: CTAs per SM (1 producer + 8 consumer warps each), 1..8 (0 = 2) */
    int32_t combine_stage_bytes;  /* TMA combine: bytes of the k row chunks per stage, multiple of 16 (0 = 16 KiB) */
    int32_t combine_unroll;       /* vector combine: 16-byte loads per lane and slot per step, 1..8
                                     (0 = 2 for k <= 2, 1 for k = 4, 4 for k = 8; the slots are then taken
                                     in groups sized for about 4 loads per lane) */
    int32_t recv_order;           /* A2AV_ORDER_SOURCE (0) or A2AV_ORDER_EXPERT */
} a2av_config_t;

/* Caller-owned device arrays the split counts and offsets are written to
 * (layouts above).  They are GPU-resident outputs: the host never needs them
 * for the data path. */
typedef struct {
    int32_t *send_counts;
    int32_t *send_offsets;
    int32_t *recv_counts;
    int32_t *recv_offsets;
    int32_t *recv_expert_counts;
    int32_t *recv_total;
    int32_t *window_base;
    int32_t *recv_expert_offsets; /* [R][R][Epr]; required with A2AV_ORDER_EXPERT, else may be NULL (not written) */
} a2av_splits_t;

/* Host-only check of a configuration against the limits above; touches no GPU. */
a2av_status_t a2av_config_check(const a2av_config_t *cfg);

/* Rows the recv arena needs: R*T*k (packed), R*window_rows (fixed) or
 * R*R*T*k (padded); -1 for an invalid configuration.  Host-only. */
int64_t a2av_recv_arena_rows(const a2av_config_t *cfg);

/* Create a plan: validates `cfg`, allocates the plan's small device
 * workspace (per-tile counts, completion counters, status word) on
 * cfg->device and sets kernel attributes.  Synchronous; not capturable.
 * Call it once, outside graph capture, and reuse the plan. */
a2av_status_t a2av_plan_create(const a2av_config_t *cfg, a2av_plan_t *out_plan);

/* Free the plan's workspace.  The caller must have finished all work
 * enqueued with it.  NULL is accepted. */
a2av_status_t a2av_plan_destroy(a2av_plan_t plan);

/* Dispatch = a2av_splits followed by a2av_pack on `stream` (two kernels).
 * Counts the routing on the device (the counts never go to the host), scans
 * them into send/recv splits and window bases, and stores every token row
 * x[s][t] once per routed expert straight into its destination window:
 * recv[slot_map[s][t][j]] = x[s][t].  Only routed rows move; rows of the
 * arena beyond each window's recv_total are left untouched.  recv must not
 * overlap x.  [Inference section and Figure 13; digest 3.3: the counts are
 * taken from device memory at execution time, nothing is padded, and the
 * received counts are handed back -- here in splits.] */
a2av_status_t a2av_dispatch(a2av_plan_t plan, const void *x, const int32_t *topk_idx,
                            const a2av_splits_t *splits, void *recv, int32_t *slot_map, void *stream);

/* First half of dispatch (one kernel): per-rank expert histogram with a
 * fused device-side scan.  Fills every array of `splits` and leaves in
 * slot_map an intermediate per-assignment rank that a2av_pack consumes
 * (slot_map is final only after a2av_pack).  [Digest 3.3 and the Inference
 * section: counts made and kept on the GPU; the received counts are part of
 * the result.] */
a2av_status_t a2av_splits(a2av_plan_t plan, const int32_t *topk_idx, const a2av_splits_t *splits,
                          int32_t *slot_map, void *stream);

/* Second half of dispatch (one kernel): pack + exchange.  Must follow
 * a2av_splits with the same topk_idx, splits and slot_map on the same
 * stream.  Writes recv rows and the final slot_map. */
a2av_status_t a2av_pack(a2av_plan_t plan, const void *x, const int32_t *topk_idx,
                        const a2av_splits_t *splits, void *recv, int32_t *slot_map, void *stream);

/* Combine (one kernel): out[s][t] = bf16_rne(sum_{j=0..k-1, slot>=0}
 * gate_w[s][t][j] * y[slot_map[s][t][j]]), fp32 accumulation from 0 in slot
 * order with separately rounded products and sums.  y has the recv layout
 * (the expert outputs written in place of, or beside, the received rows).
 * out must not overlap y.  [Deep dive section 7, Figure 13: the token
 * shuffle is followed by the combine.] */
a2av_status_t a2av_combine(a2av_plan_t plan, const void *y, const float *gate_w, const int32_t *slot_map,
                           void *out, void *stream);

/* Expert stand-in used by checkable workloads (not part of the collective):
 * for every assignment with slot >= 0, y[slot] = bf16_rne(float(recv[slot]) *
 * (1 + e/E)), e its global expert id, computed in fp32 (e/E, then 1 + that,
 * then the product).  y may equal recv (in place). */
a2av_status_t a2av_expert_scale(a2av_plan_t plan, const void *recv, const int32_t *topk_idx,
                                const int32_t *slot_map, void *y, void *stream);

/* Dispatch that allocates nothing (no plan, no cudaMalloc, no allocating
 * library call).  The paper has no counterpart.  It is for callers that
 * cannot allocate device memory where they dispatch: code inside a framework
 * whose caching allocator owns all device memory and must not be bypassed,
 * processes under a fixed device-memory budget that is spent by the time
 * this library runs, and latency-critical loops that cannot take the
 * implicit device synchronisation of cudaMalloc.  Same inputs, outputs and
 * results as a2av_dispatch on a plan made from `cfg`; the scratch the splits
 * and pack kernels need lives in one static device array of the library
 * (1 MiB per GPU that loads the library, held until process exit), which
 * bounds the shapes it accepts: R*ceil(T*k/2048)*E + R + (R + 1) int32 (each
 * term rounded up to 64) must fit in 262144, else A2AV_ERR_INVALID_ARG with
 * the sizes in a2av_last_error().  `dev_status` is a caller-owned device
 * uint32 that the kernels OR the A2AV_DEV_* bits into (the caller clears it).
 * The first call on each device does a one-time set-up with that device
 * current (it looks up the array's device address, a synchronous runtime
 * call, and sets the kernels' attributes), and the first call with each
 * configuration computes its launch shapes; both are kept for later calls,
 * so make the first call before any stream capture.  cudaDeviceReset after
 * the first call is not supported (the address looked up would belong to the
 * destroyed context).  Every call uses the same array and leaves its last
 * contents there (the counters that must start at zero are cleared on the
 * stream by each call): calls that overlap on the GPU -- on different
 * streams, or from different threads without ordering -- race on it. */
a2av_status_t a2av_dispatch_static(const a2av_config_t *cfg, const void *x, const int32_t *topk_idx,
                                   const a2av_splits_t *splits, void *recv, int32_t *slot_map,
                                   uint32_t *dev_status, void *stream);

/* The padded baseline (plans with window_mode A2AV_WINDOW_PADDED): what an
 * AllToAllv whose counts are frozen at graph capture has to do.  The counts
 * cannot be trusted when the collective runs, so every source sends the
 * worst case -- every token to one expert, T*k rows -- to every destination
 * and most of what moves is padding [Inference section; digest 3.3; the
 * deep dive, Figure 15].  Three steps on `stream`:
 *   a2av_splits          counts and scans as usual; recv_offsets[d][s] = s*T*k,
 *                        window_base[d] = d*R*T*k; slot_map gets the padded rows
 *   a2av_pack_padded     the sort into the send buffer: sendbuf[(s*R + d)*T*k + p]
 *                        = the p-th row rank s sends to d (expert order); rows past
 *                        the real count are left as they are (padding)
 *   a2av_exchange_padded the fixed-size AllToAll: for every (s, d) all T*k rows of
 *                        sendbuf's segment (s, d) go to recv's segment (d, s),
 *                        padding included
 * sendbuf and recv are bf16 [R*R*T*k][H] (a2av_recv_arena_rows), distinct and
 * disjoint from x.  a2av_combine then works unchanged.  a2av_dispatch and
 * a2av_pack reject padded plans. */
a2av_status_t a2av_dispatch_padded(a2av_plan_t plan, const void *x, const int32_t *topk_idx,
                                   const a2av_splits_t *splits, void *sendbuf, void *recv, int32_t *slot_map,
                                   void *stream);
a2av_status_t a2av_pack_padded(a2av_plan_t plan, const void *x, const int32_t *topk_idx,
                               const a2av_splits_t *splits, void *sendbuf, int32_t *slot_map, void *stream);
a2av_status_t a2av_exchange_padded(a2av_plan_t plan, const void *sendbuf, void *recv, void *stream);

/* Router (one kernel): for every token, topk_idx[s][t][0..k-1] = the k
 * experts with the largest logits[s][t][.] (fp32 [R][T][E], device), in
 * descending order, equal logits by lower expert id, a NaN logit counted as
 * -infinity; gate_w[s][t][j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the
 * selected logits (fp32, sum in slot order; 1/k each if every selected
 * logit is -infinity).  Tokens that take no part (a2av_set_active_tokens)
 * are left untouched.  Needs k <= E.  Its outputs feed a2av_dispatch /
 * a2av_combine.
 * [Inference section, Figure 13: a router kernel picks each token's experts
 * before the tokens are sorted by expert; the pages do not define it.] */
a2av_status_t a2av_route(a2av_plan_t plan, const float *logits, int32_t *topk_idx, float *gate_w, void *stream);

/* The router and the first half of dispatch: the same routing as a2av_route
 * (written to topk_idx and gate_w) and the same splits and slot_map contents
 * as a2av_splits.  By default it enqueues exactly those two kernels.  With
 * A2AV_FLAG_ROUTE_FUSED in the plan's flags, and when k divides 32 and
 * E <= 256, it is one kernel instead: the tiled histogram kernel routes the
 * tokens of its own tiles and counts the ids as it chooses them, without
 * reading topk_idx back.  (Measured on GB300 the fused kernel is slower: a
 * histogram tile of 2048 assignments gives the routing too few warps.)
 * Follow it with a2av_pack on the same plan and stream, as after
 * a2av_splits.  Same argument rules as those two calls; needs k <= E.
 * [Inference section, Figure 13: the router kernel picks the experts, and the
 * tokens are then sorted and counted by expert.] */
a2av_status_t a2av_route_splits(a2av_plan_t plan, const float *logits, int32_t *topk_idx, float *gate_w,
                                const a2av_splits_t *splits, int32_t *slot_map, void *stream);

/* Variable batches (decode): from now on every kernel this plan enqueues
 * reads num_tokens[s] -- a caller-owned DEVICE array of R int32, read when
 * the kernel runs, so it may change between replays of a captured graph --
 * and only tokens t < num_tokens[s] of rank s take part (values are clamped
 * to [0, T]).  Tokens that take no part are not counted, not copied, get
 * slot -1 without a bad-id status, and their `out` rows are left untouched
 * by a2av_combine.  NULL (the default) makes every token take part.  Host
 * call, no device work; affects later enqueues only.  [Inference section:
 * the real counts change with every routing while the captured graph stays
 * the same; buffers keep their worst-case size and consecutive calls use
 * alternating receive buffers (double buffering).] */
a2av_status_t a2av_set_active_tokens(a2av_plan_t plan, const int32_t *num_tokens);

/* Diagnostic hook for the failure path of the bounded waits (not part of
 * the method).  The TMA pack (default), the TMA combine
 * (A2AV_FLAG_COMBINE_TMA) and the lane-per-token router (a2av_route's
 * default) wait on mbarriers for the bulk copies they issued
 * themselves; each wait gives up after a bounded number of polls, sets
 * A2AV_DEV_WAIT_TIMEOUT in the status word and ends the CTA in order (it
 * first lets every copy it issued land, with the full bound).  This call sets
 * the main-loop limit of those waits for later enqueues on `plan`: polls >= 0
 * polls at most that many times (0 gives up at once, which makes the
 * give-up path run on purpose; the rows, or the routing, of that call are
 * then incomplete),
 * polls < 0 restores the default (2^22 polls, seconds: never reached while
 * the copies work).  Values above the default are clamped to it.  Host call,
 * no device work.  [No counterpart on the pages: the pages' collectives
 * time out on the host; here every device wait reports through the status
 * word instead of hanging.] */
a2av_status_t a2av_set_wait_limit(a2av_plan_t plan, int64_t polls);

/* Copy the device status word to *bits (synchronises `stream`); if `clear`,
 * reset it to 0 afterwards.  Not capturable. */
a2av_status_t a2av_read_device_status(a2av_plan_t plan, uint32_t *bits, int clear, void *stream);

/* Device address of the plan's 32-bit status word, for callers that read it
 * themselves (for instance inside their own graph). */
const void *a2av_device_status_ptr(a2av_plan_t plan);

/* Number of kernels the plan has enqueued (or had captured) so far. */
int64_t a2av_plan_launches(a2av_plan_t plan);

/* Static text for a status value. */
const char *a2av_status_string(a2av_status_t status);

/* Text of the last CUDA error seen by this library on the calling thread
 * (empty if none). */
const char *a2av_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* A2AV_H */
