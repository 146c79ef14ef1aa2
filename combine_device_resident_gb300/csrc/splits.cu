// Routing histogram + device-side scan: the split counts of a MoE AllToAllv
// computed and kept on the GPU.
//
// NCCLX (Section 6.1), pages: abhik.ai, section on inference (the counts come
// out of GPU work and must not be copied to the host; the collective hands
// back the counts it received) and the hungchun0201 digest, 3.3
// AllToAllvDynamic (the counts are taken from device memory at execution
// time).  Order inside a window: expert, then token, then slot -- a stable
// sort by expert, as the pages' send buffer is ordered by expert.
//
// Two kernels; the plan picks one.
//
// Cluster kernel (R <= 16 ranks, T*k <= 8192): one CTA per rank, the R CTAs
// form one thread-block cluster.  CTA s counts rank s, scans its counts in
// shared memory, and writes its count to every window straight into the
// shared memory of every other CTA (distributed shared memory); after the
// next cluster barrier each CTA holds all R x R counts and derives the
// receive offsets and window bases itself.  (The expert receive order also
// needs every rank's per-expert counts, which it reads from the peers'
// shared memory instead.)  It then writes the final arena row of each of its
// assignments into slot_map.  No global atomics, fences, or waits beyond the
// hardware cluster barrier.
//
// Tiled kernel (any shape): grid (tiles, R), one tile of kHistTile
// assignments per CTA.  The last CTA of a rank to finish (atomic ticket, no
// waiting) scans that rank's tile counts; the last rank to finish computes
// the cross-rank part.  slot_map then holds each assignment's rank inside its
// tile and the pack kernel assembles the final row from the splits arrays.
// Tickets are re-armed by the CTA that consumed them, so the kernel can be
// replayed from a CUDA graph.
//
// Both count with warp aggregation: a warp handles 32 consecutive
// assignments per round; the lanes holding the same expert find each other
// with one ballot per bit of the expert id, their group does one
// shared-memory update, and each lane gets its stable rank in the group.
// Both let the pack kernel begin launching as soon as the kernel before
// them has completed (programmatic dependent launch), so the pack streams x
// in while they work; it waits for this grid before reading their output.
//
// Compile-time variants: with or without the code that fills
// recv_expert_offsets (the first row of each (source, local expert) block;
// chosen per launch from whether the caller passed that array), the cluster
// kernel per receive order, and a routed instantiation of the tiled kernel
// (A2AV_FLAG_ROUTE_FUSED: each warp routes its own tokens from the logits
// and counts the ids it chose, 32 warps of 2 rounds per tile).
#include "a2av_internal.cuh"
#include "route_select.cuh"

namespace a2av {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive scan, in place, of n ints in shared memory; returns the total.
// `wtot` is shared scratch of at least 33 ints.  All threads must call it.
__device__ int block_exclusive_scan(int *buf, int n, int *wtot) {
    const int nt = blockDim.x, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += buf[i];
    const int incl = warp_inclusive_scan(sum, lane);
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nw ? wtot[lane] : 0;
        const int iv = warp_inclusive_scan(v, lane);
        if (lane < nw) wtot[lane] = iv - v;
        if (lane == 31) wtot[32] = iv;
    }
    __syncthreads();
    int run = wtot[warp] + incl - sum;
    for (int i = lo; i < hi; ++i) {
        const int v = buf[i];
        buf[i] = run;
        run += v;
    }
    const int total = wtot[32];
    __syncthreads();
    return total;
}

// One round of warp-aggregated counting: lane's assignment has expert `e`
// (valid when `good`); `cnt` is this warp's per-expert counter row.  Returns
// the lane's stable rank among the warp's assignments of its expert so far.
__device__ __forceinline__ int count_round(int *cnt, int e, bool good, int E, int key_bits) {
    const uint32_t peers = peers_by_ballot(good ? (uint32_t)e : (uint32_t)E, key_bits);
    const int before = __popc(peers & lanemask_lt());
    const int c = good ? cnt[e] : 0;
    __syncwarp();
    if (good && before == 0) cnt[e] = c + __popc(peers);
    __syncwarp();
    return c + before;
}

// ---------------------------------------------------------------------------
// Tiled kernel
// ---------------------------------------------------------------------------
// WRITE_REO: fill splits.recv_expert_offsets (compile-time: a caller that
// does not ask for them gets a kernel without that code -- measured: the
// mere presence of the extra stores in these latency-bound kernels cost about
// 1 us per call).  ROUTE_EPL > 0: the router runs here -- each warp routes the
// tokens of its assignments from the logits (route_token, ROUTE_EPL logits
// per lane), writes topk_idx and gate_w, and counts the ids it just chose,
// without reading topk_idx back (needs k | 32).  NW warps per CTA, ROUNDS
// rounds of 32 assignments per warp: one tile = NW * 32 * ROUNDS.
template <bool WRITE_REO, int ROUTE_EPL, int NW>
__global__ void __launch_bounds__(NW * 32) hist_scan_kernel(const HistArgs a) {
    constexpr int ROUNDS = kHistTile / (NW * 32);
    static_assert(NW * 32 * ROUNDS == kHistTile, "a CTA covers one tile");
    extern __shared__ int smem[];
    __shared__ int wtot[33];
    __shared__ int last;
    const Geometry &g = a.g;
    const int E = g.E, R = g.R, epr = g.epr, ES = E + 1;  // ES: padded row stride
    const int s = blockIdx.y, tile = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int A = g.T * g.k;  // assignments of one rank

    // ---- per-warp counts of this tile --------------------------------------
    int *cnt = smem + warp * ES;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    // On few-token calls launched as a programmatic dependent of whatever
    // kernel came before (the previous call's combine, a router): nothing
    // global is read or written before its grid has completed, num_tokens
    // included.
    grid_dependency_wait();
    // The pack kernel (a programmatic dependent) may launch now.  Not
    // earlier: the pack loads x before its own dependency wait, and x may be
    // the output of the kernel just waited for (the previous call's out).
    grid_launch_dependents();
    const int As = active_tokens(a.num_tokens, s, g.T) * g.k;  // assignments taking part
    const int w0 = tile * kHistTile + warp * (32 * ROUNDS);
    int key[ROUNDS], rank[ROUNDS];
    int vals[ROUNDS];
    if (ROUTE_EPL == 0) {
        const int32_t *idx = a.idx + (size_t)s * A;
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int ai = w0 + r * 32 + lane;
            vals[r] = ai < A ? __ldg(idx + ai) : -1;
        }
    } else {
        // a round of 32 assignments is 32/k whole tokens; lane l counts slot
        // l % k of token l / k
        const int k = g.k, tpr = 32 / k, lt = lane / k, ls = lane - lt * k;
        const int Ts = active_tokens(a.num_tokens, s, g.T);
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            vals[r] = -1;
            const int t0 = (w0 + r * 32) / k;
            for (int m = 0; m < tpr; ++m) {
                const int t = t0 + m;
                if (t >= Ts) break;  // warp-uniform: past the rank's active (or all) tokens
                int32_t id;
                float w;
                const size_t tok = (size_t)s * g.T + t;
                route_token<(ROUTE_EPL > 0 ? ROUTE_EPL : 1)>(a.logits + tok * E, E, k, lane, id, w);
                if (lane < k) {
                    a.idx_out[tok * k + lane] = id;
                    a.gate_out[tok * k + lane] = w;
                }
                const int got = __shfl_sync(kFull, id, ls);
                if (lt == m) vals[r] = got;
            }
        }
    }
    bool bad = false;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        if (w0 + r * 32 >= A) break;  // warp-uniform
        const int ai = w0 + r * 32 + lane;
        const int e = vals[r];
        const bool inr = ai < As;
        const bool good = inr && e >= 0 && e < E;
        bad |= inr && !good;
        rank[r] = count_round(cnt, e, good, E, g.key_bits);
        key[r] = good ? e : -1;
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_BAD_EXPERT);
    __syncthreads();

    // ---- scan over warps: warp bases and the tile's per-expert counts -------
    int32_t *tb = a.tile_base + ((size_t)s * g.tiles + tile) * E;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int v = smem[w * ES + e];
            smem[w * ES + e] = run;
            run += v;
        }
        tb[e] = run;
    }
    __syncthreads();
    int32_t *sm = a.slot_map + (size_t)s * A;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        if (w0 + r * 32 >= A) break;
        const int ai = w0 + r * 32 + lane;
        if (ai < A) sm[ai] = key[r] >= 0 ? cnt[key[r]] + rank[r] : -1;
    }

    // ---- last CTA of rank s: scan tiles, per-rank splits ----------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&a.counters[s], 1u) == (uint32_t)(g.tiles - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();

    int *tot = smem;  // E ints
    constexpr int kTileRegs = 16;
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t *col = a.tile_base + (size_t)s * g.tiles * E + e;
        int run = 0;
        for (int t0 = 0; t0 < g.tiles; t0 += kTileRegs) {
            int v[kTileRegs];
#pragma unroll
            for (int q = 0; q < kTileRegs; ++q) v[q] = t0 + q < g.tiles ? __ldcg(col + (size_t)(t0 + q) * E) : 0;
#pragma unroll
            for (int q = 0; q < kTileRegs; ++q) {
                if (t0 + q < g.tiles) __stcg(col + (size_t)(t0 + q) * E, run);
                run += v[q];
            }
        }
        tot[e] = run;
        a.sp.send_counts[(size_t)s * E + e] = run;
        const int d = e / epr, le = e - d * epr;
        a.sp.recv_expert_counts[((size_t)d * R + s) * epr + le] = run;
    }
    __syncthreads();
    const int valid = block_exclusive_scan(tot, E, wtot);
    for (int e = tid; e < E; e += blockDim.x) a.sp.send_offsets[(size_t)s * E + e] = tot[e];
    if (tid == 0) {
        a.rank_total[s] = valid;
        a.counters[s] = 0;  // re-arm for the next call
    }

    // ---- last rank: cross-rank splits and window bases ------------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&a.counters[R], 1u) == (uint32_t)(R - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();

    // recv_counts[d][src] = send_offsets[src][(d+1)*epr] - send_offsets[src][d*epr]
    // (the end of the last window is the source's count of valid assignments)
    int *rc = smem;          // [R][R]
    int *wt = smem + R * R;  // [R] window totals
    const int32_t *so = a.sp.send_offsets;
    constexpr int kPairRegs = 16;
    for (int p0 = tid * kPairRegs; p0 < R * R; p0 += blockDim.x * kPairRegs) {
        int hi[kPairRegs], lo[kPairRegs];
#pragma unroll
        for (int q = 0; q < kPairRegs; ++q) {
            const int p = p0 + q;
            const int d = p / R, src = p - d * R;
            lo[q] = p < R * R ? __ldcg(so + (size_t)src * E + d * epr) : 0;
            hi[q] = p < R * R ? (d + 1 < R ? __ldcg(so + (size_t)src * E + (d + 1) * epr) : __ldcg(a.rank_total + src))
                              : 0;
        }
#pragma unroll
        for (int q = 0; q < kPairRegs; ++q)
            if (p0 + q < R * R) rc[p0 + q] = hi[q] - lo[q];
    }
    __syncthreads();
    // one warp per window: receive offsets (scan over sources) and totals
    for (int d = warp; d < R; d += NW) {
        int carry = 0;
        for (int c0 = 0; c0 < R; c0 += 32) {
            const int src = c0 + lane;
            const int v = src < R ? rc[d * R + src] : 0;
            const int incl = warp_inclusive_scan(v, lane);
            if (src < R) {
                a.sp.recv_counts[d * R + src] = v;
                a.sp.recv_offsets[d * R + src] =
                    g.window_mode == A2AV_WINDOW_PADDED ? (int)((long long)src * g.T * g.k) : carry + incl - v;
            }
            carry += __shfl_sync(kFull, incl, 31);
        }
        if (lane == 0) {
            wt[d] = carry;
            a.sp.recv_total[d] = carry;
        }
    }
    __syncthreads();
    if (warp == 0) {
        const bool fixed = g.window_mode == A2AV_WINDOW_FIXED;
        int carry = 0;
        bool ovf = false;
        for (int c0 = 0; c0 < R; c0 += 32) {
            const int d = c0 + lane;
            const int v = d < R ? wt[d] : 0;
            const int incl = warp_inclusive_scan(v, lane);
            if (d < R)
                a.sp.window_base[d] = fixed ? (int)((long long)d * g.window_rows)
                                    : g.window_mode == A2AV_WINDOW_PADDED ? (int)((long long)d * R * g.T * g.k)
                                                                           : carry + incl - v;
            ovf |= fixed && d < R && v > g.window_rows;
            carry += __shfl_sync(kFull, incl, 31);
        }
        if (__any_sync(kFull, ovf) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
        if (lane == 0) a.counters[R] = 0;  // re-arm
    }

    // ---- first row of every (source, local expert) block ----------------------
    // One warp per destination d: d's received counts rec[d][s][le] (E
    // contiguous ints) are staged in the warp's scratch and scanned there.
    if (!WRITE_REO) return;
    int32_t *reo = a.sp.recv_expert_offsets;
    int *buf = smem + R * R + R + warp * E;  // [E] per warp
    const bool padded = g.window_mode == A2AV_WINDOW_PADDED;
    for (int d = warp; d < R; d += NW) {
        const int32_t *rec = a.sp.recv_expert_counts + (size_t)d * E;  // [R][epr]
        for (int i = lane; i < E; i += 32) buf[i] = __ldcg(rec + i);
        __syncwarp();
        int32_t *out = reo + (size_t)d * E;
        int carry = 0;
        if (g.recv_order == A2AV_ORDER_EXPERT) {
            // lane = local expert: its block starts after the lower experts'
            // rows (all sources); inside it the sources follow in order
            for (int l0 = 0; l0 < epr; l0 += 32) {
                const int le = l0 + lane;
                int tot = 0;
                if (le < epr)
                    for (int src = 0; src < R; ++src) tot += buf[src * epr + le];
                const int incl = warp_inclusive_scan(tot, lane);
                int run = carry + incl - tot;
                if (le < epr)
                    for (int src = 0; src < R; ++src) {
                        out[src * epr + le] = run;
                        run += buf[src * epr + le];
                    }
                carry += __shfl_sync(kFull, incl, 31);
            }
        } else {
            // lane = source: its segment start, then its rows for the lower
            // local experts
            for (int s0 = 0; s0 < R; s0 += 32) {
                const int src = s0 + lane;
                const int v = src < R ? rc[d * R + src] : 0;
                const int incl = warp_inclusive_scan(v, lane);
                if (src < R) {
                    int run = padded ? (int)((long long)src * g.T * g.k) : carry + incl - v;
                    for (int le = 0; le < epr; ++le) {
                        out[src * epr + le] = run;
                        run += buf[src * epr + le];
                    }
                }
                carry += __shfl_sync(kFull, incl, 31);
            }
        }
        __syncwarp();  // the scratch is refilled for the next destination
    }
}

size_t hist_smem_bytes(const Geometry &g, bool write_reo, int nw) {
    const size_t a = (size_t)nw * (g.E + 1), b = (size_t)g.R * g.R + g.R + (write_reo ? (size_t)nw * g.E : 0);
    return sizeof(int) * (a > b ? a : b);
}

// The routed tiled kernel: 32 warps of 2 rounds per tile (more warps in
// flight for the routing work), E <= 32 * 8, k dividing 32.
constexpr int kRoutedWarps = 32;
constexpr int kRoutedMaxEpl = 8;
int routed_epl(const Geometry &g) {
    if (g.k < 1 || 32 % g.k != 0 || g.k > g.E) return 0;
    const int need = (g.E + 31) / 32;
    return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= kRoutedMaxEpl ? 8 : 0;
}

// ---------------------------------------------------------------------------
// Cluster kernel
// ---------------------------------------------------------------------------
constexpr int kClusterWarps = 32;
constexpr int kClusterThreads = kClusterWarps * 32;
constexpr int kClusterRounds = 8;  // rounds of 32 assignments per warp
constexpr int kClusterMaxRanks = 16;

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_smem(const int *p, int rank) {
    const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}
__device__ __forceinline__ int ld_dsmem(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_dsmem(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// BY_EXPERT: the expert-grouped receive order; WRITE_REO: fill
// splits.recv_expert_offsets.  Both compile-time, so the plain source-order
// instantiation carries none of their work.
template <bool BY_EXPERT, bool WRITE_REO>
__global__ void __launch_bounds__(kClusterThreads, 1) splits_cluster_kernel(const HistArgs a) {
    extern __shared__ int smem[];
    const Geometry &g = a.g;
    const int R = g.R, E = g.E, epr = g.epr, ES = E + 1;
    const int A = g.T * g.k;
    const int s = blockIdx.x;  // == rank of this CTA in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = ((A + kClusterWarps - 1) / kClusterWarps + 31) / 32 * 32;
    const int a0 = warp * chunk;
    int *cnt = smem;                    // [32][E+1] per-warp counts -> warp bases
    int *so = cnt + kClusterWarps * ES;  // [E + 1] send offsets of this rank (so[E] = total)
    int *rc = so + (E + 1);              // [R][R] recv counts, [d][src]
    int *ro = rc + R * R;                // [R] receive offset of this rank in window d
    int *wb = ro + R;                    // [R] window totals, then bases
    int *xb = wb + R;                    // [E] expert order: rows of expert e on ranks below s
    int *xt = xb + E;                    // [E] expert order: rows of e on all ranks, then e's block start
    constexpr bool by_expert = BY_EXPERT;
    // On few-token calls launched as a programmatic dependent of the kernel
    // before it (the previous call's combine, a router): it is resident early
    // and reads or writes nothing global before that grid has completed.  Meanwhile it
    // asks L2 for its routing lines (a prefetch only warms L2, which stays
    // coherent with the predecessor's writes; the values are loaded after the
    // wait) and clears its counters.
    const int32_t *idx = a.idx + (size_t)s * A;
#pragma unroll
    for (int r = 0; r < kClusterRounds; ++r) {
        const int ai = a0 + r * 32 + lane;
        if (r * 32 < chunk && ai < A && (lane & 31) == 0) prefetch_l2(idx + ai);
    }
    for (int i = tid; i < kClusterWarps * ES; i += kClusterThreads) cnt[i] = 0;
    if (by_expert)
        for (int i = tid; i < 2 * E; i += kClusterThreads) xb[i] = 0;  // xb and xt
    grid_dependency_wait();
    grid_launch_dependents();  // the pack may launch now (as in hist_scan_kernel)
    const int As = active_tokens(a.num_tokens, s, g.T) * g.k;  // assignments taking part
    int vals[kClusterRounds];
#pragma unroll
    for (int r = 0; r < kClusterRounds; ++r) {
        const int ai = a0 + r * 32 + lane;
        vals[r] = (r * 32 < chunk && ai < A) ? __ldg(idx + ai) : -1;
    }
    __syncthreads();

    int key[kClusterRounds], rank[kClusterRounds];
    int *mine = cnt + warp * ES;
    {
        bool bad = false;
#pragma unroll
        for (int r = 0; r < kClusterRounds; ++r) {
            if (r * 32 >= chunk || a0 + r * 32 >= A) break;  // warp-uniform
            const int ai = a0 + r * 32 + lane;
            const bool inr = ai < As;
            const int e = vals[r];
            const bool good = inr && e >= 0 && e < E;
            bad |= inr && !good;
            rank[r] = count_round(mine, e, good, E, g.key_bits);
            key[r] = good ? e : -1;
        }
        if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_BAD_EXPERT);
    }
    __syncthreads();

    // per expert, one warp: scan the 32 warps' counts (lane = warp index)
    for (int e = warp; e < E; e += kClusterWarps) {
        const int v = cnt[lane * ES + e];
        const int incl = warp_inclusive_scan(v, lane);
        cnt[lane * ES + e] = incl - v;
        if (lane == 31) so[e] = incl;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the E counts by one warp (one barrier, not four)
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += so[i];
        const int incl = warp_inclusive_scan(sum, lane);
        int run = incl - sum;
        for (int i = lo; i < hi; ++i) {
            const int v = so[i];
            so[i] = run;
            run += v;
        }
        if (lane == 31) so[E] = incl;
    }
    __syncthreads();
    // (send_counts, send_offsets and recv_expert_counts are stored after the
    // cluster barriers: a barrier's release would otherwise wait for them)

    if (!by_expert) {
        // Push: this rank's count to every window d goes into rc[d][s] of
        // every peer CTA, so no remote load sits between the two barriers.
        // The first makes sure every peer CTA has started (its shared memory
        // may be written); nothing reads a peer's shared memory after the
        // second.
        cluster_barrier();
        for (int p = tid; p < R * R; p += kClusterThreads) {
            const int peer = p / R, d = p - peer * R;
            st_dsmem(peer_smem(rc + d * R + s, peer), so[(d + 1) * epr] - so[d * epr]);
        }
        // the release makes the pushes visible to every peer's acquire; it
        // also orders this CTA's own threads (rc is read by other warps below)
        cluster_barrier();
    } else {
        // every rank's send offsets are now in its CTA's shared memory
        cluster_barrier();
        for (int p = tid; p < R * R; p += kClusterThreads) {
            const int d = p / R, src = p - d * R;
            rc[p] = ld_dsmem(peer_smem(so + (d + 1) * epr, src)) - ld_dsmem(peer_smem(so + d * epr, src));
        }
        // one (source, expert) pair per thread, summed with shared-memory atomics
        for (int p = tid; p < R * E; p += kClusterThreads) {
            const int src = p / E, e = p - src * E;
            const int c = ld_dsmem(peer_smem(so + e + 1, src)) - ld_dsmem(peer_smem(so + e, src));
            if (c) {
                atomicAdd(&xt[e], c);
                if (src < s) atomicAdd(&xb[e], c);
            }
        }
        // no CTA may leave (or reuse) its shared memory until every peer has
        // read it; the barrier also orders this CTA's own threads
        cluster_barrier();
    }

    // one warp per window: this rank's receive offset and the window total
    if (warp < R) {
        const int d = warp;
        const int v = lane < R ? rc[d * R + lane] : 0;
        const int incl = warp_inclusive_scan(v, lane);
        if (lane == s) {
            const int off = g.window_mode == A2AV_WINDOW_PADDED ? (int)((long long)s * g.T * g.k) : incl - v;
            ro[d] = off;
            a.sp.recv_counts[d * R + s] = v;
            a.sp.recv_offsets[d * R + s] = off;
        }
        if (lane == 31) {
            wb[d] = incl;
            if (s == 0) a.sp.recv_total[d] = incl;
        }
    }
    __syncthreads();
    if (warp == 0) {
        const int v = lane < R ? wb[lane] : 0;
        const int incl = warp_inclusive_scan(v, lane);
        const bool fixed = g.window_mode == A2AV_WINDOW_FIXED;
        const long long base = fixed ? (long long)lane * g.window_rows
                               : g.window_mode == A2AV_WINDOW_PADDED ? (long long)lane * R * g.T * g.k
                                                                      : (long long)(incl - v);
        const bool ovf = fixed && lane < R && v > g.window_rows;
        if (s == 0 && __any_sync(kFull, ovf) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
        __syncwarp();
        if (lane < R) {
            wb[lane] = (int)base;
            if (s == 0) a.sp.window_base[lane] = (int)base;
        }
    }
    if (by_expert)  // block start of each expert: scan of the totals over its window's experts
        for (int d = warp; d < R; d += kClusterWarps) {
            int carry = 0;
            for (int c0 = 0; c0 < epr; c0 += 32) {
                const int le = c0 + lane;
                const int v = le < epr ? xt[d * epr + le] : 0;
                const int incl = warp_inclusive_scan(v, lane);
                if (le < epr) xt[d * epr + le] = carry + incl - v;
                carry += __shfl_sync(kFull, incl, 31);
            }
        }
    __syncthreads();

    bool ovf = false;
    int32_t *sm = a.slot_map + (size_t)s * A;
#pragma unroll
    for (int r = 0; r < kClusterRounds; ++r) {
        if (r * 32 >= chunk || a0 + r * 32 >= A) break;  // warp-uniform
        const int ai = a0 + r * 32 + lane;
        if (ai < A) {
            int32_t row = -1;
            const int e = key[r];
            if (e >= 0) {
                const int d = e / epr;
                const long long rel = (by_expert ? (long long)xt[e] + xb[e] : (long long)ro[d] + so[e] - so[d * epr]) +
                                      mine[e] + rank[r];
                if (g.window_mode == A2AV_WINDOW_FIXED && rel >= g.window_rows)
                    ovf = true;
                else
                    row = (int32_t)(wb[d] + rel);
            }
            sm[ai] = row;
        }
    }
    if (__any_sync(kFull, ovf) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
    // this rank's send counts and offsets (so[] holds the exclusive offsets, so[E] the total)
    for (int e = tid; e < E; e += kClusterThreads) {
        const int c = so[e + 1] - so[e];
        const int d = e / epr, le = e - d * epr;
        a.sp.send_counts[(size_t)s * E + e] = c;
        a.sp.send_offsets[(size_t)s * E + e] = so[e];
        a.sp.recv_expert_counts[((size_t)d * R + s) * epr + le] = c;
    }
    // first row of each of this rank's (destination, local expert) blocks
    if (WRITE_REO)
        for (int e = tid; e < E; e += kClusterThreads) {
            const int d = e / epr, le = e - d * epr;
            a.sp.recv_expert_offsets[((size_t)d * R + s) * epr + le] =
                by_expert ? xt[e] + xb[e] : ro[d] + so[e] - so[d * epr];
        }
}

size_t cluster_smem_bytes(const Geometry &g) {
    return sizeof(int) * ((size_t)kClusterWarps * (g.E + 1) + (g.E + 1) + (size_t)g.R * g.R + 2 * (size_t)g.R +
                          (g.recv_order == A2AV_ORDER_EXPERT ? 2 * (size_t)g.E : 0));
}

bool cluster_eligible(const Geometry &g) {
    if (g.R > kClusterMaxRanks) return false;
    const long long A = (long long)g.T * g.k;
    const long long chunk = ((A + kClusterWarps - 1) / kClusterWarps + 31) / 32 * 32;
    return chunk <= 32 * kClusterRounds && cluster_smem_bytes(g) <= 160 * 1024;
}

using SplitsKernel = void (*)(const HistArgs);
// (the expert order always writes the offsets: the pack reads them)
SplitsKernel cluster_kernel_for(const Geometry &g, bool write_reo) {
    if (g.recv_order == A2AV_ORDER_EXPERT) return splits_cluster_kernel<true, true>;
    return write_reo ? splits_cluster_kernel<false, true> : splits_cluster_kernel<false, false>;
}
SplitsKernel hist_kernel_for(bool write_reo, int route_epl = 0) {
    switch (route_epl) {
        case 1: return write_reo ? hist_scan_kernel<true, 1, kRoutedWarps> : hist_scan_kernel<false, 1, kRoutedWarps>;
        case 2: return write_reo ? hist_scan_kernel<true, 2, kRoutedWarps> : hist_scan_kernel<false, 2, kRoutedWarps>;
        case 4: return write_reo ? hist_scan_kernel<true, 4, kRoutedWarps> : hist_scan_kernel<false, 4, kRoutedWarps>;
        case 8: return write_reo ? hist_scan_kernel<true, 8, kRoutedWarps> : hist_scan_kernel<false, 8, kRoutedWarps>;
        default: return write_reo ? hist_scan_kernel<true, 0, kHistWarps> : hist_scan_kernel<false, 0, kHistWarps>;
    }
}

// `at` holds two attributes: the cluster shape and (when `pdl`) the
// programmatic stream serialization the kernels' grid_dependency_wait needs.
cudaLaunchConfig_t cluster_launch_config(const a2av_plan_s &p, cudaLaunchAttribute *at, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(p.g.R);
    lc.blockDim = dim3(kClusterThreads);
    lc.dynamicSmemBytes = cluster_smem_bytes(p.g);
    lc.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.g.R;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = pdl ? 2 : 1;
    return lc;
}

// The tiled kernels' launch: grid (tiles, R), a programmatic dependent of
// the kernel before it when `pdl`.
cudaError_t launch_tiled(SplitsKernel k, const a2av_plan_s &p, int threads, size_t smem, const HistArgs &a,
                         cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(p.g.tiles, p.g.R);
    lc.blockDim = dim3(threads);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k, a);
}

// Whether a splits kernel starts as a programmatic dependent of the kernel
// before it.  Only on few-token calls, where the overlap is worth a
// microsecond or two of a ~20 us step.  On large calls it is worth nothing,
// and it has a cost: its CTAs, placed while that kernel still holds most
// SMs, crowd onto the few SMs with room.  Then the persistent pack grid
// launched after them cannot seat all its CTAs, and those left over run a
// whole pack-length second wave (measured with the router letting its
// dependents launch early: r32 E256 top-8 step 2,654 -> 3,926 us).
bool splits_pdl(const a2av_plan_s &p) { return p.few_tokens; }

}  // namespace

// Per-kernel caps shared by every plan: the largest any valid plan needs.
cudaError_t configure_tiled_hist_attributes() {
    Geometry worst{};
    worst.R = kMaxRanks;
    worst.E = kMaxExperts;
    Geometry worst_routed = worst;
    worst_routed.E = 32 * kRoutedMaxEpl;
    cudaError_t e = cudaSuccess;
    for (bool w : {false, true}) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(hist_kernel_for(w), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)hist_smem_bytes(worst, true, kHistWarps));
        for (int epl : {1, 2, 4, 8})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(hist_kernel_for(w, epl), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)hist_smem_bytes(worst_routed, true, kRoutedWarps));
    }
    return e;
}

cudaError_t configure_hist(a2av_plan_s &p) {
    {  // the tiled kernels serve every plan (the routed one even cluster-eligible ones)
        cudaError_t e = configure_tiled_hist_attributes();
        if (e != cudaSuccess) return e;
    }
    if (!(p.cfg.flags & A2AV_FLAG_SPLITS_TILED) && cluster_eligible(p.g)) {
        cudaError_t e = cudaSuccess;
        for (auto k : {splits_cluster_kernel<false, false>, splits_cluster_kernel<false, true>,
                       splits_cluster_kernel<true, true>}) {
            if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
        if (e != cudaSuccess) return e;
        const auto kern = cluster_kernel_for(p.g, true);
        // Can a cluster of R such CTAs be resident at all on this device?
        cudaLaunchAttribute at[2];
        cudaLaunchConfig_t lc = cluster_launch_config(p, at, nullptr, false);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &lc);
        if (e == cudaSuccess && clusters >= 1) {
            p.splits_small = 1;
            p.hist.block = kClusterThreads;
            p.hist.smem = cluster_smem_bytes(p.g);
            p.hist.grid = p.g.R;
            return cudaSuccess;
        }
        cudaGetLastError();  // not resident as a cluster here: use the tiled kernel
    }
    p.splits_small = 0;
    p.hist.block = kHistThreads;
    p.hist.smem = hist_smem_bytes(p.g, true, kHistWarps);  // launches without the offsets take less
    p.hist.grid = p.g.tiles;
    return cudaSuccess;
}

cudaError_t launch_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s) {
    const bool reo = a.sp.recv_expert_offsets != nullptr;
    cudaError_t e;
    if (p.splits_small) {
        cudaLaunchAttribute at[2];
        cudaLaunchConfig_t lc = cluster_launch_config(p, at, s, splits_pdl(p));
        e = cudaLaunchKernelEx(&lc, cluster_kernel_for(p.g, reo), a);
    } else {
        e = launch_tiled(hist_kernel_for(reo), p, kHistThreads, hist_smem_bytes(p.g, reo, kHistWarps), a, s,
                         splits_pdl(p));
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace a2av

namespace a2av {

bool routed_splits_supported(const a2av_plan_s &p) { return routed_epl(p.g) != 0; }

// The router fused into the tiled histogram: always the tiled kernel, so
// slot_map holds tile ranks afterwards (the pack assembles the rows).
cudaError_t launch_routed_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s) {
    const int epl = routed_epl(p.g);
    if (!epl) return cudaErrorInvalidValue;
    const bool reo = a.sp.recv_expert_offsets != nullptr;
    cudaError_t e = launch_tiled(hist_kernel_for(reo, epl), p, kRoutedWarps * 32,
                                 hist_smem_bytes(p.g, reo, kRoutedWarps), a, s, splits_pdl(p));
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace a2av
