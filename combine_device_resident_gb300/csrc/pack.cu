// Fused pack + exchange: every token row x[s][t] is read once and stored
// straight into the destination window of each of its k experts, at the row
// its stable expert order gives it.  No send buffer, no padding: only routed
// rows move, from the caller's buffer straight into the caller's windows
// (NCCLX pages: the abhik.ai sections on CTran's zero-copy transfers and on
// inference; the hungchun0201 digest, 3.3 AllToAllvDynamic).
//
// Row of assignment (s, t, j) with expert e on rank d = e / (E/R):
//   rel = recv_offsets[d][s] + send_offsets[s][e] - send_offsets[s][d*E/R]
//         + tile_base[s][tile(t*k+j)][e] + rank_in_tile
//   (expert-grouped receive order: rel = recv_expert_offsets[d][s][e - d*E/R]
//    + tile_base[s][tile(t*k+j)][e] + rank_in_tile)
//   row = window_base[d] + rel        (dropped if rel >= window_rows, fixed mode)
// (all produced on the device by the splits kernel; with the cluster splits
// kernel slot_map already holds the row).
//
// Two variants:
//   * TMA bulk (default): persistent grid, one warp per CTA.  Row chunks are
//     brought into a ring of shared-memory stages by cp.async.bulk
//     (completion on an mbarrier) and written out by k cp.async.bulk stores,
//     one per destination row; the ring keeps many KB in flight per SM with a
//     single issuing thread.  Lanes compute the destination rows of the next
//     batch of tokens while the copies run.  The CTAs split the tokens that
//     take part (per-rank active counts), so variable batches stay balanced.
//   * LSU: warp per token, 16-byte vector loads (no L1 allocation) and stores.
#include "a2av_internal.cuh"

namespace a2av {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
__device__ __forceinline__ long long arena_rows_of(const Geometry &g) {
    const long long tk = (long long)g.T * g.k;
    return g.window_mode == A2AV_WINDOW_FIXED ? (long long)g.R * g.window_rows
           : g.window_mode == A2AV_WINDOW_PADDED ? (long long)g.R * g.R * tk
                                                  : (long long)g.R * tk;
}

// Padded plans store into the padded send buffer: the row a receive-side
// (window d, segment s, position p) row came from, (s*R + d)*T*k + p; -1 if
// the row does not lie in source s's segment (never for rows the splits
// kernel produced; the store is then skipped).
__device__ __forceinline__ long long send_row_of(const PackArgs &a, long long row, int s) {
    const long long tk = a.padded_tk, window = (long long)a.g.R * tk;
    const long long d = row / window;
    const long long p = row - d * window - (long long)s * tk;
    if (p < 0 || p >= tk) return -1;
    return ((long long)s * a.g.R + d) * tk + p;
}

// Final arena row of assignment j of flat token `tok`, or -1 if dropped.  With
// the tiled splits kernel slot_map holds the rank inside the histogram tile
// and the row is assembled here; with the one-CTA kernel it is already final.
__device__ __forceinline__ int32_t final_row(const PackArgs &a, long long tok, int j, uint32_t &ovf) {
    const Geometry &g = a.g;
    const size_t ga = (size_t)tok * g.k + j;
    if (a.rows_final) {
        const int32_t row = a.slot_map[ga];
        if (row >= arena_rows_of(g)) {
            ovf = 1;
            return -1;
        }
        return row;
    }
    const int e = __ldg(a.idx + ga);
    const int r = a.slot_map[ga];
    if (e < 0 || e >= g.E || r < 0) return -1;
    const int s = (int)(tok / g.T);
    const int t = (int)(tok - (long long)s * g.T);
    const int tl = (t * g.k + j) / kHistTile;
    const int d = e / g.epr;
    // rank of the assignment among rank s's rows for expert e, plus where
    // that (s, e) block starts in window d
    const long long in_block = (long long)__ldg(a.tile_base + ((size_t)s * g.tiles + tl) * g.E + e) + r;
    const long long rel =
        in_block + (g.recv_order == A2AV_ORDER_EXPERT
                        ? (long long)__ldg(a.recv_expert_offsets + ((size_t)d * g.R + s) * g.epr + (e - d * g.epr))
                        : (long long)__ldg(a.recv_offsets + (size_t)d * g.R + s) +
                              __ldg(a.send_offsets + (size_t)s * g.E + e) -
                              __ldg(a.send_offsets + (size_t)s * g.E + (size_t)d * g.epr));
    const long long cap = g.window_mode == A2AV_WINDOW_FIXED ? g.window_rows : (long long)g.R * g.T * g.k;
    // (packed: a window holds at most R*T*k rows; padded: a window is R*T*k rows)
    if (rel < 0 || rel >= cap) {
        ovf = 1;
        return -1;
    }
    const long long row = (long long)__ldg(a.window_base + d) + rel;
    if (row < 0 || row >= arena_rows_of(g)) {
        ovf = 1;
        return -1;
    }
    return (int32_t)row;
}

// Shared memory after the NS stages: NS stage barriers, prefix [R + 1].
__host__ __device__ constexpr size_t pack_tail_bytes(int stages) {
    return (size_t)stages * 8 + 4 * (size_t)(kMaxRanks + 1);
}

// One warp per CTA; lane 0 keeps the chunk loads in flight and issues the k
// stores of every chunk, the lanes compute the destination rows of the next
// batch of BT = 32/k tokens (lane l: token l / k, slot l % k).  COUNTED:
// per-rank active token counts (a.num_tokens); PADDED: stores go to the
// padded send buffer; STREAM: the row stores carry an evict-first L2 policy
// (plans whose rows cannot stay in L2 until the combine and whose pack is
// write-dominated, see configure_pack).  All compile-time, so the plain
// instantiation keeps the shortest issue loop (measured: the issuing lane's
// scalar work between copy-engine waits shows up directly in the kernel's
// time).
template <bool COUNTED, bool PADDED, bool STREAM>
__global__ void __launch_bounds__(32, 1) pack_tma_kernel(const PackArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    // Latency-bound calls (few tokens): the combine, a programmatic
    // dependent, may take its SM slots now; its own grid-dependency wait
    // still covers every store of this grid.  Not on large calls: there the
    // early CTAs cost the pack about 4% (r16 E128 T4096 top-2: 661 against
    // 636 us per step).
    if (a.trigger_early) grid_launch_dependents();
    const Geometry &g = a.g;
    const int lane = threadIdx.x;
    const int NS = a.stages, CH = a.chunk_bytes, nch = a.nchunks;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)NS * CH);
    int *prefix = reinterpret_cast<int *>(bars + NS);  // [R + 1] tokens taking part before rank s

    // The CTAs split the tokens that take part, not all R*T: with per-rank
    // counts the active tokens are the first num_tokens[s] of every rank, and
    // contiguous ranges of all tokens would leave most CTAs idle.  Active
    // index ia maps to rank s (prefix[s] <= ia < prefix[s+1]) and token
    // ia - prefix[s]; without counts the map is the identity.
    if (COUNTED) {
        int carry = 0;
        for (int c0 = 0; c0 < g.R; c0 += 32) {
            const int s = c0 + lane;
            const int v = s < g.R ? active_tokens(a.num_tokens, s, g.T) : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += t;
            }
            if (s < g.R) prefix[s] = carry + incl - v;
            carry += __shfl_sync(kFull, incl, 31);
        }
        if (lane == 0) prefix[g.R] = carry;
        __syncwarp();
    }
    const long long nact = COUNTED ? (long long)prefix[g.R] : (long long)g.R * g.T;
    auto token_of = [&](long long ia) -> long long {
        if (!COUNTED) return ia;
        int lo = 0, hi = g.R - 1;  // the last rank whose prefix is <= ia (skips empty ranks)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= ia) lo = mid;
            else hi = mid - 1;
        }
        return (long long)lo * g.T + (ia - prefix[lo]);
    };

    const long long per = (nact + gridDim.x - 1) / gridDim.x;
    const long long ia_b = min(nact, (long long)blockIdx.x * per);
    const long long ia_e = min(nact, ia_b + per);
    if (ia_b >= ia_e) return;
    const long long n = (ia_e - ia_b) * nch;
    const size_t rowb = (size_t)g.H * 2;
    const int BT = max(1, 32 / g.k);
    const char *x = reinterpret_cast<const char *>(a.x);
    char *recv = reinterpret_cast<char *>(a.recv);

    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Loads walk the active tokens in order: with counts, step to the next
    // token inside a rank and search only when the rank changes.
    long long l_ia = -1, l_tok = 0, l_end = 0;
    auto load_token = [&](long long ia) -> long long {
        if (!COUNTED) return ia;
        if (ia == l_ia) return l_tok;
        if (ia == l_ia + 1 && l_tok + 1 < l_end) {
            l_ia = ia;
            return ++l_tok;
        }
        l_ia = ia;
        l_tok = token_of(ia);
        const int s = (int)(l_tok / g.T);
        l_end = (long long)s * g.T + (prefix[s + 1] - prefix[s]);
        return l_tok;
    };
    // x is read exactly once: its lines go to L2 as evict-first, so the rows
    // the pack writes (read again by the combine) stay resident instead
    // (measured on r8 E16 T1024 H5120, an arena of 84 MB against the 126 MB
    // L2: step 55.4 -> 52.5 us, the combine finding its rows in L2).
    const uint64_t x_policy = l2_policy_evict_first();
    // unit p = (active token ia_b + p / nch, chunk p % nch) into stage p % NS
    auto issue_load = [&](long long p) {
        const long long tok = load_token(ia_b + p / nch);
        const uint32_t off = (uint32_t)(p % nch) * CH;
        const uint32_t bytes = (uint32_t)min((size_t)CH, rowb - off);
        uint64_t *bar = &bars[p % NS];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load_hint(smem + (size_t)(p % NS) * CH, x + (size_t)tok * rowb + off, bytes, bar, x_policy);
    };
    // Store rows of the batch starting at active index ib0; slot_map gets the
    // arena row, padded plans store into the padded send buffer instead.
    auto rows_of_batch = [&](long long ib0, uint32_t &ovf) -> int32_t {
        const int b = lane / g.k, j = lane - b * g.k;
        if (b >= BT || ib0 + b >= ia_e) return -1;
        const long long tok = token_of(ib0 + b);
        const int32_t row = final_row(a, tok, j, ovf);
        if (!a.rows_final) a.slot_map[(size_t)tok * g.k + j] = row;
        if (!PADDED || row < 0) return row;
        return (int32_t)send_row_of(a, row, (int)(tok / g.T));
    };
    // Loads may run NS - LAG units ahead; up to LAG store groups may still be
    // reading their stage when the next load is issued.
    const int LAG = a.lag;
    const long long pre = min(n, (long long)NS);
    if (lane == 0)
        for (long long p = 0; p < pre; ++p) issue_load(p);
    long long issued = pre;  // loads issued so far (units 0..issued-1)

    // x does not depend on the splits kernel; everything below does.  (The
    // splits kernels let this grid launch only once the kernel before them
    // has completed, so these loads never race with a kernel writing x: the
    // previous call's combine, when its out is this call's x.)
    grid_dependency_wait();

    uint32_t ovf = 0;
    long long ib0 = ia_b;
    int32_t cur = rows_of_batch(ib0, ovf);
    int32_t nxt = rows_of_batch(ib0 + BT, ovf);
    bool timed_out = false;
    long long i = 0;
    for (; i < n; ++i) {
        const long long ia = ia_b + i / nch;
        const int c = (int)(i % nch);
        if (ia >= ib0 + BT) {
            ib0 += BT;
            cur = nxt;
            nxt = rows_of_batch(ib0 + BT, ovf);
        }
        const int st = (int)(i % NS);
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(&bars[st], (uint32_t)((i / NS) & 1), a.wait_polls);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) {
            timed_out = true;
            break;
        }
        const uint32_t off = (uint32_t)c * CH;
        const uint32_t bytes = (uint32_t)min((size_t)CH, rowb - off);
        const int lb = (int)(ia - ib0);
        if (lane == 0) fence_proxy_async_smem();
        for (int j = 0; j < g.k; ++j) {
            const int32_t rj = __shfl_sync(kFull, cur, lb * g.k + j);
            if (lane == 0 && rj >= 0) {
                if (STREAM)
                    bulk_store_hint(recv + (size_t)rj * rowb + off, smem + (size_t)st * CH, bytes, x_policy);
                else
                    bulk_store(recv + (size_t)rj * rowb + off, smem + (size_t)st * CH, bytes);
            }
        }
        if (lane == 0) {
            bulk_commit();
            const long long jdone = i - (LAG - 1);  // its stores have finished reading once <= LAG-1 groups pend
            if (jdone >= 0 && jdone + NS < n) {
                bulk_wait_read_upto(LAG - 1);
                issue_load(jdone + NS);
                issued = jdone + NS + 1;
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        // Leave once every stage has been read: the stores' writes to the
        // windows complete before the grid does, which is what the kernels
        // after it wait for.
        if (timed_out) bulk_wait_all();
        else bulk_wait_read<0>();
        if (timed_out) {
            // Leave only after every load this CTA issued has landed, unit i's
            // included (it is the one the main loop gave up on).  These waits
            // keep the full bound whatever the main loop's limit: each load is
            // a bulk copy of in-bounds rows of x, which completes in
            // microseconds unless the memory system itself has failed (then
            // the context is already lost), so the bound is never reached in a
            // live context.
            for (long long p = i; p < issued; ++p)
                mbar_wait_bounded(&bars[p % NS], (uint32_t)((p / NS) & 1), kWaitLimit);
            atomicOr(a.status, kDevWaitTimeout);
        }
    }
    if (__any_sync(kFull, ovf != 0) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
}

template <int U>
__global__ void __launch_bounds__(256) pack_lsu_kernel(const PackArgs a) {
    const Geometry &g = a.g;
    const int lane = threadIdx.x & 31;
    const long long ntok = (long long)g.R * g.T;
    const int nv = g.H >> 3;
    const size_t rowb = (size_t)g.H * 2;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    uint32_t ovf = 0;
    if (a.trigger_early) grid_launch_dependents();  // as in the TMA pack
    grid_dependency_wait();
    for (long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < ntok; u += nw) {
        const int s_tok = (int)(u / g.T);
        if (u - (long long)s_tok * g.T >= active_tokens(a.num_tokens, s_tok, g.T)) continue;  // warp-uniform
        int32_t row = -1;
        if (lane < g.k) {
            row = final_row(a, u, lane, ovf);
            if (!a.rows_final) a.slot_map[(size_t)u * g.k + lane] = row;
        }
        const char *src = reinterpret_cast<const char *>(a.x) + (size_t)u * rowb;
        for (int vb = 0; vb < nv; vb += 32 * U) {
            uint4 buf[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int v = vb + q * 32 + lane;
                if (v < nv) buf[q] = ld_stream_v4(src + (size_t)v * 16);
            }
            for (int j = 0; j < g.k; ++j) {
                const int32_t rj = __shfl_sync(kFull, row, j);
                if (rj < 0) continue;
                const long long drow = a.padded_tk ? send_row_of(a, rj, s_tok) : (long long)rj;
                if (drow < 0) continue;
                char *dst = reinterpret_cast<char *>(a.recv) + (size_t)drow * rowb;
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const int v = vb + q * 32 + lane;
                    if (v < nv) st_v4(dst + (size_t)v * 16, buf[q]);
                }
            }
        }
    }
    if (__any_sync(kFull, ovf != 0) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
}

constexpr int kLsuUnroll = 4;
constexpr size_t kTmaChunkMax = 16384;
constexpr int kDefaultCtasPerSm = 4;
constexpr int kDefaultLag = 2;

}  // namespace

namespace {
// The fixed-size AllToAll of the padded baseline: every (source s,
// destination d) segment of T*k rows, padding included, from the send buffer
// at (s*R + d) to the receive arena at (d*R + s).  16-byte vectors, four in
// flight per thread, grid-stride over the whole arena.
__global__ void __launch_bounds__(256) exchange_padded_kernel(const ExchangeArgs a) {
    grid_dependency_wait();
    const long long total = (long long)a.R * a.R * a.block_vecs;
    const long long nthr = (long long)gridDim.x * blockDim.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.sendbuf);
    uint4 *dst = reinterpret_cast<uint4 *>(a.recv);
    for (long long v0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; v0 < total; v0 += 4 * nthr) {
        uint4 buf[4];
        long long from[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const long long v = v0 + q * nthr;
            from[q] = -1;
            if (v < total) {
                const long long blk = v / a.block_vecs, in = v - blk * a.block_vecs;
                const long long d = blk / a.R, s = blk - d * a.R;
                from[q] = (s * a.R + d) * a.block_vecs + in;
                buf[q] = ld_stream_v4(src + from[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (from[q] >= 0) st_v4(dst + v0 + q * nthr, buf[q]);
    }
}
}  // namespace

cudaError_t configure_pack(a2av_plan_s &p) {
    const size_t rowb = (size_t)p.g.H * 2;
    {
        // Evict-first row stores: when the rows a call writes cannot stay in
        // L2 until the combine and the pack is write-dominated (k >= 4).
        // Measured, L2 flushed: r32 E256 T2048 H7168 top-8 pack 1,346 ->
        // 1,326 us, step 2,652 -> 2,627 us; r16 E128 T4096 top-2 pack
        // unchanged (317 us) while the combine in the step lost 4.5 us (it
        // finds fewer of the last rows in L2); the hinted store with the
        // normal policy on L2-sized calls cost r8 E128 T256 0.15 us.
        int l2 = 0;
        cudaError_t e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, p.cfg.device);
        if (e != cudaSuccess) return e;
        p.pack_stream_rows = p.g.k >= 4 && (double)p.g.R * p.g.T * p.g.k * (double)rowb > (double)l2 ? 1 : 0;
    }
    {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, exchange_padded_kernel, 256, 0);
        if (e != cudaSuccess) return e;
        p.exchange.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
        p.exchange.block = 256;
    }
    if (!p.pack_tma) {
        p.pack.block = 256;
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pack_lsu_kernel<kLsuUnroll>, 256, 0);
        if (e != cudaSuccess) return e;
        p.pack.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
        p.pack.smem = 0;
        return cudaSuccess;
    }
    const int ctas_per_sm = p.cfg.pack_ctas_per_sm > 0 ? p.cfg.pack_ctas_per_sm : kDefaultCtasPerSm;
    // Defaults measured on GB300: for k >= 4 small stages (many loads ahead)
    // and a deep store lag; for k <= 2 whole-row stages (big stores per unit).
    const bool wide = p.g.k >= 4;
    size_t chunk = p.cfg.pack_stage_bytes > 0 ? (size_t)p.cfg.pack_stage_bytes : (wide ? 2048 : kTmaChunkMax);
    chunk = (chunk + 15) / 16 * 16;
    if (chunk > rowb) chunk = rowb;
    int max_optin = 0, per_sm = 0, reserved = 0;
    cudaError_t e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.cfg.device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p.cfg.device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, p.cfg.device);
    if (e != cudaSuccess) return e;
    // ctas_per_sm CTAs share the SM's shared memory, each with the runtime's
    // per-block reservation on top of its dynamic size
    size_t budget = (size_t)per_sm / ctas_per_sm;
    budget = budget > (size_t)reserved ? budget - reserved : 0;
    if (budget > (size_t)max_optin) budget = max_optin;
    const size_t tail0 = pack_tail_bytes(0);  // prefix
    budget = budget > tail0 ? budget - tail0 : budget;
    // at least two stages: shrink the chunk if the requested one does not fit
    while (chunk > 256 && 2 * (chunk + 8) > budget) chunk = (chunk / 2 + 15) / 16 * 16;
    const int nch2 = (int)((rowb + chunk - 1) / chunk);
    int stages = (int)((budget) / (chunk + 8));
    if (stages > 32) stages = 32;
    int lag = p.cfg.pack_store_lag > 0 ? p.cfg.pack_store_lag : (wide ? 6 : kDefaultLag);
    if (lag > stages - 1) lag = stages - 1;
    if (lag < 1) return cudaErrorInvalidConfiguration;
    p.pack_lag = lag;
    p.pack_chunk_bytes = (int32_t)chunk;
    p.pack_nchunks = nch2;
    p.pack_stages = stages;
    p.pack.block = 32;
    p.pack.smem = (size_t)stages * chunk + pack_tail_bytes(stages);
    p.pack.grid = p.num_sms * ctas_per_sm;
    // The attribute is a per-kernel cap shared by every plan: raise it to the
    // device maximum (never lower it to this plan's size).
    for (auto kern : {pack_tma_kernel<false, false, false>, pack_tma_kernel<false, true, false>,
                      pack_tma_kernel<true, false, false>, pack_tma_kernel<true, true, false>,
                      pack_tma_kernel<false, false, true>, pack_tma_kernel<false, true, true>,
                      pack_tma_kernel<true, false, true>, pack_tma_kernel<true, true, true>}) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}


cudaError_t launch_exchange_padded(const a2av_plan_s &p, const ExchangeArgs &a, cudaStream_t s) {
    cudaError_t e = launch_pdl(exchange_padded_kernel, p.exchange.grid, 256, 0, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pack(const a2av_plan_s &p, const PackArgs &a, cudaStream_t s) {
    PackArgs b = a;  // b.rows_final: set by the caller from the splits launch that preceded it
    b.trigger_early = p.few_tokens ? 1 : 0;
    b.wait_polls = p.wait_polls;
    cudaError_t e;
    if (p.pack_tma) {
        b.chunk_bytes = p.pack_chunk_bytes;
        b.nchunks = p.pack_nchunks;
        b.stages = p.pack_stages;
        b.lag = p.pack_lag;
        const bool counted = b.num_tokens != nullptr, padded = b.padded_tk != 0;
        auto kern = p.pack_stream_rows
                        ? (counted ? (padded ? pack_tma_kernel<true, true, true> : pack_tma_kernel<true, false, true>)
                                   : (padded ? pack_tma_kernel<false, true, true> : pack_tma_kernel<false, false, true>))
                        : (counted ? (padded ? pack_tma_kernel<true, true, false> : pack_tma_kernel<true, false, false>)
                                   : (padded ? pack_tma_kernel<false, true, false>
                                             : pack_tma_kernel<false, false, false>));
        e = launch_pdl(kern, p.pack.grid, p.pack.block, p.pack.smem, s, b);
    } else {
        e = launch_pdl(pack_lsu_kernel<kLsuUnroll>, p.pack.grid, p.pack.block, 0, s, b);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace a2av
