/*
 * a2av_oracle.c -- plain, slow, single-threaded CPU oracle of the MoE
 * AllToAllvDynamic data plane (dispatch, then top-k weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path calls this file:
 * only the tests, the smoke check and the benchmark's CPU baseline / reference
 * arm load it.  It shares no code, header, table or constant with the CUDA
 * library; both sides only consume the same seeded inputs.
 *
 * Source: NCCLX, "Collective Communication for 100k+ GPUs" (Meta), as
 * described on the pages
 *   [P1] abhik.ai/papers/ncclx, section "Inference: small messages, unknown
 *        sizes" (Figure 13 pipeline; Section 6.1 AllToAllvDynamic);
 *   [P2] hungchun0201 research digest, section 3.3 "AllToAllvDynamic";
 *   [P3] qiguanping.github.io deep dive, section 7 (Figure 13, dispatch
 *        shuffle and combine; Figures 16-17, GPU-resident metadata).
 * What the pages fix:
 *   - a router chooses the experts of each token; the tokens are sorted by
 *     expert into a send buffer; an AllToAllv sends each one to the rank
 *     that holds its expert [P1, Inference, Figure 13];
 *   - the split counts are computed on the GPU and read from GPU memory when
 *     the collective runs; only real tokens are sent, no padding to the
 *     worst case [P1 Inference; P2 3.3];
 *   - the collective returns the counts it received [P1 Inference];
 *   - the tokens come back and are combined [P3 section 7, Figure 13].
 * Readings where the pages are silent (each is stated again where used):
 *   R1  expert e lives on rank e / (E/R)   (contiguous blocks of E/R experts);
 *   R2  the sort by expert is stable: expert ascending, then token t,
 *       then slot j;
 *   R3  the AllToAllv convention: window d holds the segments of sources
 *       0..R-1 back to back, in source order, with no gaps;
 *   R4  windows: "packed" mode places window d right after window d-1 in one
 *       arena; "fixed" mode gives window d the rows [d*W, (d+1)*W);
 *       "padded" mode is the worst-case layout a host-side AllToAllv must
 *       use under graph capture [P1 Inference; P2 3.3]: every (source,
 *       destination) pair gets T*k rows, so window d starts at d*R*T*k and
 *       source s's segment inside it at s*T*k;
 *   R5  combine: out = bf16_rne( sum_j w_j * y[slot(t,j)] ), accumulated in
 *       fp32 from 0.0f in slot order j = 0..k-1, each product and each sum
 *       rounded on its own (this file must be built with -ffp-contract=off);
 *   R7  variable batches: when a per-rank count num_tokens[s] is given, only
 *       tokens t < num_tokens[s] of rank s take part (the others are not
 *       counted, get slot -1 and no combine output) -- the counts change from
 *       step to step while the buffers stay sized for T [P1 Inference;
 *       P3 section 7, double buffering];
 *   R8  the router (top-k of per-token logits, softmax gates): see
 *       oracle_route below;
 *   R9  receive order: the AllToAllv convention (R3) leaves window d in
 *       source order, and inside each source's segment the rows are sorted by
 *       expert.  The expert-grouped view is the same window regrouped so that
 *       each local expert's rows are contiguous, the step after the exchange
 *       that feeds one GEMM per expert [P1 Inference, Figure 13: the received
 *       tokens go to their experts' FFN].  Reading: window d holds local
 *       expert 0's rows, then local expert 1's, and so on; inside an expert,
 *       source 0's rows, then source 1's, each in the order its segment had
 *       (token, then slot).  The counts are those of the source order; only
 *       the places differ.  Selected by ORACLE_ORDER_EXPERT in window_mode;
 *       not defined for the padded layout;
 *   R6  error handling: an expert id outside [0, E) is dropped (not counted,
 *       slot -1, status bit 0); in fixed mode a row whose window-relative
 *       position is >= W is dropped (slot -1, status bit 1) while the counts
 *       still report the routed totals; combine skips slot -1.
 *
 * Layouts (all row-major, C order):
 *   x          uint16 bf16 bits  [R][T][H]
 *   idx        int32             [R][T][k]
 *   gate       float32           [R][T][k]
 *   send_counts, send_offsets    int32 [R][E]
 *   recv_counts, recv_offsets    int32 [R][R]      (destination-major: [d][s])
 *   recv_expert_counts           int32 [R][R][E/R] ([d][s][local expert])
 *   recv_expert_offsets          int32 [R][R][E/R] ([d][s][local expert]):
 *                                window-relative first row of the rows
 *                                source s sends to local expert le of rank d
 *   recv_total, window_base      int32 [R]
 *   recv, y    uint16 bf16 bits  [rows][H]
 *   slot_map   int32             [R][T][k]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_EXPERT 1u
#define ORACLE_WINDOW_OVERFLOW 2u
/* window_mode = layout (0 packed, 1 fixed, 2 padded) | receive order (R9) */
#define ORACLE_ORDER_EXPERT 0x100
#define ORACLE_LAYOUT(m) ((m) & 0xff)

/* ---- bf16 <-> fp32 (bf16 = top 16 bits of an IEEE binary32) ---------------- */

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even, on the 16 discarded bits; NaN stays NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* Number of tokens of rank s that take part (R7): all T when no counts are
 * given, else num_tokens[s] clamped to [0, T]. */
static int active_tokens(const int32_t *num_tokens, int s, int T)
{
    if (!num_tokens)
        return T;
    int n = num_tokens[s];
    return n < 0 ? 0 : (n > T ? T : n);
}

/* ---- step 1: the split counts (what the router's counts are) ---------------
 * send_counts[s][e] = number of (t, j) on rank s with idx = e.
 * send_offsets[s][e] = sum over e' < e of send_counts[s][e']: the start of
 * expert e's block in rank s's expert-sorted send buffer (R2).
 * recv_counts[d][s] = sum of send_counts[s][e] over the experts e of rank d
 * (R1): the counts rank d receives, i.e. the transpose of the per-rank send
 * counts summed over d's experts [P1 Inference: the collective hands back
 * the counts it received].  recv_offsets[d][s] = sum over s' < s of recv_counts[d][s'] (R3).
 * recv_expert_counts[d][s][le] = send_counts[s][d*(E/R) + le].
 * recv_total[d] = sum over s of recv_counts[d][s].
 * window_base[d] = sum over d' < d of recv_total[d'] (packed) or d*W (fixed).
 * Padded mode (R4): recv_offsets[d][s] = s*T*k and window_base[d] = d*R*T*k,
 * the fixed places of the worst-case segments.
 * Returns the status bits.
 */
uint32_t oracle_splits(int R, int E, int T, int k, int window_mode, int64_t window_rows,
                       const int32_t *num_tokens, const int32_t *idx,
                       int32_t *send_counts, int32_t *send_offsets,
                       int32_t *recv_counts, int32_t *recv_offsets,
                       int32_t *recv_expert_counts, int32_t *recv_total,
                       int32_t *window_base)
{
    uint32_t status = 0;
    int epr = E / R;
    window_mode = ORACLE_LAYOUT(window_mode);
    for (int s = 0; s < R; ++s) {
        int32_t *cnt = send_counts + (size_t)s * E;
        for (int e = 0; e < E; ++e)
            cnt[e] = 0;
        int Ts = active_tokens(num_tokens, s, T);
        for (int t = 0; t < Ts; ++t)
            for (int j = 0; j < k; ++j) {
                int32_t e = idx[((size_t)s * T + t) * k + j];
                if (e < 0 || e >= E) {
                    status |= ORACLE_BAD_EXPERT;
                    continue;
                }
                cnt[e] += 1;
            }
        int32_t run = 0;
        for (int e = 0; e < E; ++e) {
            send_offsets[(size_t)s * E + e] = run;
            run += cnt[e];
        }
    }
    for (int d = 0; d < R; ++d) {
        int32_t run = 0;
        for (int s = 0; s < R; ++s) {
            int32_t c = 0;
            for (int le = 0; le < epr; ++le) {
                int32_t v = send_counts[(size_t)s * E + d * epr + le];
                recv_expert_counts[((size_t)d * R + s) * epr + le] = v;
                c += v;
            }
            recv_counts[(size_t)d * R + s] = c;
            recv_offsets[(size_t)d * R + s] = run;
            run += c;
        }
        recv_total[d] = run;
        if (window_mode == 1 && (int64_t)run > window_rows)
            status |= ORACLE_WINDOW_OVERFLOW;
    }
    int64_t base = 0;
    for (int d = 0; d < R; ++d) {
        if (window_mode == 1)
            window_base[d] = (int32_t)((int64_t)d * window_rows);
        else if (window_mode == 2)
            window_base[d] = (int32_t)((int64_t)d * R * T * k);
        else
            window_base[d] = (int32_t)base;
        base += recv_total[d];
    }
    if (window_mode == 2)
        for (int d = 0; d < R; ++d)
            for (int s = 0; s < R; ++s)
                recv_offsets[(size_t)d * R + s] = (int32_t)((int64_t)s * T * k);
    return status;
}

/* ---- where each (source, local expert) block starts in its window -----------
 * Source order (R3): source s's segment starts at recv_offsets[d][s] and is
 * sorted by expert, so its rows for local expert le start after its rows for
 * the lower local experts:
 *   recv_offsets[d][s] + sum over le' < le of recv_expert_counts[d][s][le'].
 * Expert order (R9): all rows of the lower local experts come first, then the
 * rows of expert le from the lower sources:
 *   sum over le' < le, all s' of recv_expert_counts[d][s'][le']
 *     + sum over s' < s of recv_expert_counts[d][s'][le].
 */
void oracle_recv_expert_offsets(int R, int E, int window_mode, const int32_t *recv_offsets,
                                const int32_t *recv_expert_counts, int32_t *recv_expert_offsets)
{
    int epr = E / R;
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < R; ++s)
            for (int le = 0; le < epr; ++le) {
                int64_t v = 0;
                if (window_mode & ORACLE_ORDER_EXPERT) {
                    for (int l2 = 0; l2 < le; ++l2)
                        for (int s2 = 0; s2 < R; ++s2)
                            v += recv_expert_counts[((size_t)d * R + s2) * epr + l2];
                    for (int s2 = 0; s2 < s; ++s2)
                        v += recv_expert_counts[((size_t)d * R + s2) * epr + le];
                } else {
                    v = recv_offsets[(size_t)d * R + s];
                    for (int l2 = 0; l2 < le; ++l2)
                        v += recv_expert_counts[((size_t)d * R + s) * epr + l2];
                }
                recv_expert_offsets[((size_t)d * R + s) * epr + le] = (int32_t)v;
            }
}

/* ---- step 2: the expert sort of one rank's send buffer ---------------------
 * send_pos[t][j] = position of assignment (t, j) of rank s in its
 * expert-sorted send buffer: send_offsets[s][e] + the number of earlier
 * assignments (t', j') < (t, j) of rank s with the same expert (R2, a stable
 * counting sort by expert key) [P1 Inference, Figure 13: the send buffer is
 * ordered by expert].  Dropped ids get -1.
 */
static void send_positions(int E, int T, int Ts, int k, const int32_t *idx_s, const int32_t *send_offsets_s,
                           int32_t *running, int32_t *send_pos)
{
    for (int e = 0; e < E; ++e)
        running[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int32_t e = idx_s[(size_t)t * k + j];
            if (t >= Ts) {
                send_pos[(size_t)t * k + j] = -2; /* not taking part (R7) */
                continue;
            }
            if (e < 0 || e >= E) {
                send_pos[(size_t)t * k + j] = -1;
                continue;
            }
            send_pos[(size_t)t * k + j] = send_offsets_s[e] + running[e];
            running[e] += 1;
        }
}

/* ---- step 3: where each assignment lands -------------------------------------
 * The AllToAllv copies the segment of rank s's send buffer that holds rank d's
 * experts, [send_offsets[s][d*E/R], + recv_counts[d][s]), to window d at
 * recv_offsets[d][s] (R3, R4).  So an assignment at send position p with
 * expert e (on rank d = e / (E/R)) lands at
 *   window-relative row  rel = recv_offsets[d][s] + (p - send_offsets[s][d*E/R])
 *   arena row            window_base[d] + rel,
 * dropped in fixed mode when rel >= W (R6).  slot_map records that row.
 * Returns the status bits.
 */
uint32_t oracle_slot_map(int R, int E, int T, int k, int window_mode, int64_t window_rows,
                         const int32_t *num_tokens, const int32_t *idx, const int32_t *send_offsets,
                         const int32_t *recv_offsets, const int32_t *recv_expert_offsets,
                         const int32_t *window_base, int32_t *slot_map)
{
    uint32_t status = 0;
    int epr = E / R;
    int expert_order = (window_mode & ORACLE_ORDER_EXPERT) != 0;
    window_mode = ORACLE_LAYOUT(window_mode);
    int32_t *running = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k + 4);
    for (int s = 0; s < R; ++s) {
        const int32_t *idx_s = idx + (size_t)s * T * k;
        const int32_t *so = send_offsets + (size_t)s * E;
        send_positions(E, T, active_tokens(num_tokens, s, T), k, idx_s, so, running, pos);
        for (size_t a = 0; a < (size_t)T * k; ++a) {
            int32_t e = idx_s[a];
            int32_t *slot = slot_map + (size_t)s * T * k + a;
            if (pos[a] < 0) {
                *slot = -1;
                if (pos[a] == -1)
                    status |= ORACLE_BAD_EXPERT;
                continue;
            }
            int d = e / epr;
            int64_t rel = (int64_t)recv_offsets[(size_t)d * R + s] + (pos[a] - so[d * epr]);
            if (expert_order) /* R9: the block of (s, e), then the rank inside it */
                rel = (int64_t)recv_expert_offsets[((size_t)d * R + s) * epr + (e - d * epr)] + (pos[a] - so[e]);
            if (window_mode == 1 && rel >= window_rows) {
                *slot = -1;
                status |= ORACLE_WINDOW_OVERFLOW;
                continue;
            }
            *slot = (int32_t)(window_base[d] + rel);
        }
    }
    free(pos);
    free(running);
    return status;
}

/* ---- steps 2+3 with the payload: the dispatch ----------------------------------
 * Literally: per source rank s, build the expert-sorted send buffer (copy row
 * x[s][t] to send position p for each of its assignments), then perform the
 * AllToAllv: copy each destination's segment of the send buffer into that
 * destination's window, rows in order.  Rows whose slot is -1 are not
 * written (R6).  Also fills slot_map (as oracle_slot_map).  Returns status.
 */
static uint32_t dispatch_expert_order(int R, int E, int T, int H, int k, int layout, int64_t window_rows,
                                      const int32_t *num_tokens, const uint16_t *x, const int32_t *idx,
                                      const int32_t *send_counts, const int32_t *send_offsets,
                                      const int32_t *recv_offsets, const int32_t *window_base,
                                      uint16_t *recv, int32_t *slot_map);

/* The source-order dispatch of source ranks s_begin <= s < s_end only (each
 * source's send buffer and segments are its own; the splits are those of
 * every rank).  oracle_dispatch runs it over all ranks; a caller that splits
 * the ranks into disjoint ranges and runs each range on its own thread gets
 * the same recv and slot_map (the ranges write disjoint rows and slots). */
uint32_t oracle_dispatch_ranks(int R, int E, int T, int H, int k, int window_mode, int64_t window_rows,
                               const int32_t *num_tokens, const uint16_t *x, const int32_t *idx,
                               const int32_t *send_counts, const int32_t *send_offsets,
                               const int32_t *recv_offsets, const int32_t *window_base,
                               uint16_t *recv, int32_t *slot_map, int s_begin, int s_end);

uint32_t oracle_dispatch(int R, int E, int T, int H, int k, int window_mode, int64_t window_rows,
                         const int32_t *num_tokens, const uint16_t *x, const int32_t *idx,
                         const int32_t *send_counts, const int32_t *send_offsets,
                         const int32_t *recv_offsets, const int32_t *window_base,
                         uint16_t *recv, int32_t *slot_map)
{
    if (window_mode & ORACLE_ORDER_EXPERT)
        return dispatch_expert_order(R, E, T, H, k, ORACLE_LAYOUT(window_mode), window_rows, num_tokens, x, idx,
                                     send_counts, send_offsets, recv_offsets, window_base, recv, slot_map);
    return oracle_dispatch_ranks(R, E, T, H, k, window_mode, window_rows, num_tokens, x, idx, send_counts,
                                 send_offsets, recv_offsets, window_base, recv, slot_map, 0, R);
}

uint32_t oracle_dispatch_ranks(int R, int E, int T, int H, int k, int window_mode, int64_t window_rows,
                               const int32_t *num_tokens, const uint16_t *x, const int32_t *idx,
                               const int32_t *send_counts, const int32_t *send_offsets,
                               const int32_t *recv_offsets, const int32_t *window_base,
                               uint16_t *recv, int32_t *slot_map, int s_begin, int s_end)
{
    if (window_mode & ORACLE_ORDER_EXPERT)
        return 0xffffffffu; /* source order only */
    uint32_t status = 0;
    int epr = E / R;
    size_t row_bytes = sizeof(uint16_t) * (size_t)H;
    int32_t *running = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k + 4);
    uint16_t *sendbuf = (uint16_t *)malloc(row_bytes * (size_t)T * k + 16);
    for (int s = s_begin; s < s_end; ++s) {
        const int32_t *idx_s = idx + (size_t)s * T * k;
        const int32_t *so = send_offsets + (size_t)s * E;
        const int32_t *sc = send_counts + (size_t)s * E;
        send_positions(E, T, active_tokens(num_tokens, s, T), k, idx_s, so, running, pos);
        /* the sort: rows into the send buffer in expert order */
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                int32_t p = pos[(size_t)t * k + j];
                if (p < 0) {
                    if (p == -1)
                        status |= ORACLE_BAD_EXPERT;
                    continue;
                }
                memcpy(sendbuf + (size_t)p * H, x + ((size_t)s * T + t) * H, row_bytes);
            }
        /* the AllToAllv: one contiguous segment per destination */
        for (int d = 0; d < R; ++d) {
            int32_t seg_start = so[d * epr];
            int32_t seg_len = 0;
            for (int le = 0; le < epr; ++le)
                seg_len += sc[d * epr + le];
            int64_t rel0 = recv_offsets[(size_t)d * R + s];
            for (int32_t i = 0; i < seg_len; ++i) {
                int64_t rel = rel0 + i;
                if (window_mode == 1 && rel >= window_rows) {
                    status |= ORACLE_WINDOW_OVERFLOW;
                    break;
                }
                memcpy(recv + ((size_t)window_base[d] + (size_t)rel) * H,
                       sendbuf + ((size_t)seg_start + i) * H, row_bytes);
            }
        }
        /* where each assignment went */
        for (size_t a = 0; a < (size_t)T * k; ++a) {
            int32_t *slot = slot_map + (size_t)s * T * k + a;
            if (pos[a] < 0) {
                *slot = -1;
                continue;
            }
            int d = idx_s[a] / epr;
            int64_t rel = (int64_t)recv_offsets[(size_t)d * R + s] + (pos[a] - so[d * epr]);
            *slot = (window_mode == 1 && rel >= window_rows) ? -1 : (int32_t)(window_base[d] + rel);
        }
    }
    free(sendbuf);
    free(pos);
    free(running);
    return status;
}

/* ---- the expert-grouped receive order (R9) ------------------------------------
 * Literally: perform the source-order dispatch above into windows with no
 * capacity limit (packed, back to back), then regroup every window: for local
 * expert le = 0.. and, inside it, source s = 0.., take source s's rows for
 * expert le -- in the source-order window they are the block starting at
 * recv_offsets[d][s] + (s's rows for the lower local experts), because each
 * segment is sorted by expert -- and append them to window d.  In fixed mode
 * rows appended at position >= W are dropped (R6).  slot_map follows each
 * row to its new place.
 */
static uint32_t dispatch_expert_order(int R, int E, int T, int H, int k, int layout, int64_t window_rows,
                                      const int32_t *num_tokens, const uint16_t *x, const int32_t *idx,
                                      const int32_t *send_counts, const int32_t *send_offsets,
                                      const int32_t *recv_offsets, const int32_t *window_base,
                                      uint16_t *recv, int32_t *slot_map)
{
    int epr = E / R;
    size_t row_bytes = sizeof(uint16_t) * (size_t)H;
    int32_t *tbase = (int32_t *)calloc((size_t)R + 1, sizeof(int32_t));
    int64_t rows = 0;
    for (int d = 0; d < R; ++d) {
        tbase[d] = (int32_t)rows;
        for (int s = 0; s < R; ++s)
            for (int le = 0; le < epr; ++le)
                rows += send_counts[(size_t)s * E + d * epr + le];
    }
    uint16_t *tmp = (uint16_t *)malloc(row_bytes * (size_t)rows + 16);
    int32_t *tslot = (int32_t *)malloc(sizeof(int32_t) * (size_t)R * T * k + 4);
    int64_t *moved = (int64_t *)malloc(sizeof(int64_t) * (size_t)rows + 8);
    uint32_t status = oracle_dispatch(R, E, T, H, k, 0, 0, num_tokens, x, idx, send_counts, send_offsets,
                                      recv_offsets, tbase, tmp, tslot);
    for (int d = 0; d < R; ++d) {
        int64_t run = 0;
        for (int le = 0; le < epr; ++le)
            for (int s = 0; s < R; ++s) {
                const int32_t *sc = send_counts + (size_t)s * E + d * epr;
                int64_t start = recv_offsets[(size_t)d * R + s];
                for (int l2 = 0; l2 < le; ++l2)
                    start += sc[l2];
                for (int32_t i = 0; i < sc[le]; ++i, ++run) {
                    int64_t from = tbase[d] + start + i;
                    if (layout == 1 && run >= window_rows) {
                        moved[from] = -1;
                        status |= ORACLE_WINDOW_OVERFLOW;
                        continue;
                    }
                    memcpy(recv + ((size_t)window_base[d] + (size_t)run) * H, tmp + (size_t)from * H, row_bytes);
                    moved[from] = run;
                }
            }
    }
    for (size_t a = 0; a < (size_t)R * T * k; ++a) {
        if (tslot[a] < 0) {
            slot_map[a] = -1;
            continue;
        }
        int d = idx[a] / epr;
        int64_t r = moved[tslot[a]];
        slot_map[a] = r < 0 ? -1 : (int32_t)(window_base[d] + r);
    }
    free(moved);
    free(tslot);
    free(tmp);
    free(tbase);
    return status;
}

/* ---- the expert stand-in used by the scaled workload -------------------------
 * y[row] = bf16_rne( float(recv[row]) * (1 + e/E) ), e = the assignment's global
 * expert id, for every assignment with slot >= 0.  (1 + e/E is computed in
 * fp32: e/E then 1 + that.)  Rows that no assignment owns are left as they
 * are.
 */
void oracle_expert_scale(int E, int H, int64_t n_assign, const uint16_t *recv, const int32_t *idx,
                         const int32_t *slot_map, uint16_t *y)
{
    for (int64_t a = 0; a < n_assign; ++a) {
        int32_t row = slot_map[a];
        if (row < 0)
            continue;
        float q = (float)idx[a] / (float)E;
        float scale = 1.0f + q;
        const uint16_t *src = recv + (size_t)row * H;
        uint16_t *dst = y + (size_t)row * H;
        for (int h = 0; h < H; ++h) {
            float v = oracle_bf16_to_f32(src[h]) * scale;
            dst[h] = oracle_f32_to_bf16(v);
        }
    }
}

/* ---- step 4: the combine ---------------------------------------------------------
 * For each requested token u (a flat index s*T + t):
 *   acc = 0.0f; for j = 0..k-1 with slot >= 0:  acc = acc + (w_j * y[slot][h])
 *   out[u][h] = bf16_rne(acc)                            (R5, R6)
 * [P3 section 7, Figure 13: dispatch, experts, combine.]
 */
void oracle_combine(int H, int k, const uint16_t *y, const float *gate, const int32_t *slot_map,
                    const int64_t *tokens, int64_t n_tokens, uint16_t *out)
{
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t u = tokens[i];
        const int32_t *slots = slot_map + (size_t)u * k;
        const float *w = gate + (size_t)u * k;
        uint16_t *o = out + (size_t)i * H;
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                if (slots[j] < 0)
                    continue;
                float prod = w[j] * oracle_bf16_to_f32(y[(size_t)slots[j] * H + h]);
                acc = acc + prod;
            }
            o[h] = oracle_f32_to_bf16(acc);
        }
    }
}

/* The same sum in fp64 (exact products of bf16 x fp32 values, one rounding per
 * add in fp64), returned unrounded so tests can bound the fp32 oracle. */
void oracle_combine_f64(int H, int k, const uint16_t *y, const float *gate, const int32_t *slot_map,
                        const int64_t *tokens, int64_t n_tokens, double *out)
{
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t u = tokens[i];
        const int32_t *slots = slot_map + (size_t)u * k;
        const float *w = gate + (size_t)u * k;
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                if (slots[j] < 0)
                    continue;
                acc += (double)w[j] * (double)oracle_bf16_to_f32(y[(size_t)slots[j] * H + h]);
            }
            out[(size_t)i * H + h] = acc;
        }
    }
}

/* ---- the router in front of the dispatch ------------------------------------------
 * [P1 Inference, Figure 13: a router picks the experts of each token before
 * the tokens are sorted by expert.]  The pages do not define the router;
 * reading R8: for each token, the k largest of its E logits in descending
 * order, equal logits ordered by lower expert id first, a NaN logit counted
 * as -infinity; the gate weights are the softmax of the selected logits,
 * exp(l_j - l_0) / sum_i exp(l_i - l_0) with l_0 the largest, summed in slot
 * order.  Here in fp64 (exp of the exact differences), as the reference the
 * fp32 kernel is held to.  If every selected logit is -infinity the weights
 * are 1/k each.  Tokens past num_tokens[s] (R7) are left untouched.
 */
static double router_key(float v)
{
    return v != v ? -INFINITY : (double)v;
}

/* (a, ia) comes before (b, ib) in the selection order. */
static int router_before(double a, int ia, double b, int ib)
{
    return a > b || (a == b && ia < ib);
}

void oracle_route(int R, int T, int E, int k, const int32_t *num_tokens, const float *logits,
                  int32_t *idx, double *gate)
{
    for (int s = 0; s < R; ++s) {
        int Ts = active_tokens(num_tokens, s, T);
        for (int t = 0; t < Ts; ++t) {
            const float *l = logits + ((size_t)s * T + t) * E;
            int32_t *out_i = idx + ((size_t)s * T + t) * k;
            double *out_w = gate + ((size_t)s * T + t) * k;
            double sel[32];
            double prev_v = INFINITY;
            int prev_i = -1;
            for (int j = 0; j < k; ++j) {
                /* the first element (in selection order) after the previous pick */
                int best = -1;
                double best_v = 0.0;
                for (int e = 0; e < E; ++e) {
                    double v = router_key(l[e]);
                    if (j > 0 && !router_before(prev_v, prev_i, v, e))
                        continue;
                    if (best < 0 || router_before(v, e, best_v, best)) {
                        best = e;
                        best_v = v;
                    }
                }
                out_i[j] = best;
                sel[j] = best_v;
                prev_v = best_v;
                prev_i = best;
            }
            if (sel[0] == -INFINITY) {
                for (int j = 0; j < k; ++j)
                    out_w[j] = 1.0 / k;
                continue;
            }
            double sum = 0.0, ex[32];
            for (int j = 0; j < k; ++j) {
                ex[j] = exp(sel[j] - sel[0]);
                sum += ex[j];
            }
            for (int j = 0; j < k; ++j)
                out_w[j] = ex[j] / sum;
        }
    }
}
