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
// One kernel, grid (tiles, R).  Each CTA counts one tile of kHistTile
// assignments of rank s:
//   * every warp walks 32*kHistRounds consecutive assignments; lanes holding
//     the same expert are grouped (a peer mask built from one ballot per bit
//     of the expert id), so each group does one shared-memory update
//     (warp-aggregated counts) and each lane gets its stable rank inside the
//     warp's slice;
//   * the per-warp counts are scanned in warp order, giving every assignment
//     its stable rank inside the tile (written to slot_map for the pack
//     kernel) and the tile's per-expert counts.
// The last CTA of rank s to finish (atomic ticket, no waiting) scans the tile
// counts of that rank over tiles (tile bases), writes send_counts,
// send_offsets and recv_expert_counts; the last rank to finish computes the
// cross-rank part: recv_counts (the transpose, summed over each destination's
// experts), recv_offsets, recv_total, window_base and, per (source, expert),
// the window-relative first row dest_base.  Tickets are reset to zero by the
// CTA that consumed them, so the kernel can be replayed from a CUDA graph.
//
// Problems with R <= 16 ranks and at most 8192 assignments per rank take a
// cluster kernel instead (one CTA per rank, distributed shared memory for the
// cross-rank step), which writes each assignment's final arena row straight
// into slot_map (the pack kernel then only reads it).
//
// Both kernels let the pack kernel start launching right away (programmatic
// dependent launch); the pack kernel waits for this grid before reading
// anything it writes.
#include "a2av_internal.cuh"

namespace a2av {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

// Exclusive scan, in place, of n ints in shared memory; returns the total.
// `wtot` is shared scratch of at least 33 ints.  All threads must call it.
__device__ int block_exclusive_scan(int *buf, int n, int *wtot) {
    const int nt = blockDim.x, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += buf[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nw ? wtot[lane] : 0;
        int iv = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(kFull, iv, o);
            if (lane >= o) iv += t;
        }
        if (lane < nw) wtot[lane] = iv - v;
        if (lane == 31) wtot[32] = iv;
    }
    __syncthreads();
    int run = wtot[warp] + incl - sum;
    for (int i = lo; i < hi; ++i) {
        int v = buf[i];
        buf[i] = run;
        run += v;
    }
    const int total = wtot[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kHistThreads) hist_scan_kernel(const HistArgs a) {
    extern __shared__ int smem[];
    __shared__ int wtot[33];
    __shared__ int last;
    grid_launch_dependents();
    const Geometry &g = a.g;
    const int E = g.E, R = g.R;
    const int s = blockIdx.y, tile = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int A = g.T * g.k;  // assignments of one rank

    // ---- per-warp counts of this tile --------------------------------------
    int *cnt = smem + warp * E;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();

    const int w0 = tile * kHistTile + warp * (32 * kHistRounds);
    const int32_t *idx = a.idx + (size_t)s * A;
    int key[kHistRounds], rank[kHistRounds];
    int vals[kHistRounds];
#pragma unroll
    for (int r = 0; r < kHistRounds; ++r) {
        const int ai = w0 + r * 32 + lane;
        vals[r] = ai < A ? __ldg(idx + ai) : -1;
    }
    bool bad = false;
#pragma unroll
    for (int r = 0; r < kHistRounds; ++r) {
        const int ai = w0 + r * 32 + lane;
        const int e = vals[r];
        const bool inr = ai < A;
        const bool good = inr && e >= 0 && e < E;
        bad |= inr && !good;
        const int kk = good ? e : -1;
        const uint32_t peers = peers_by_ballot(good ? (uint32_t)e : (uint32_t)E, g.key_bits);
        const int before = __popc(peers & lanemask_lt());
        const int c = good ? cnt[e] : 0;
        __syncwarp();
        if (good && before == 0) cnt[e] = c + __popc(peers);
        __syncwarp();
        key[r] = kk;
        rank[r] = c + before;
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_BAD_EXPERT);
    __syncthreads();

    // ---- scan over warps: warp bases and the tile's per-expert counts ---------
    int32_t *tb = a.tile_base + ((size_t)s * g.tiles + tile) * E;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kHistWarps; ++w) {
            const int v = smem[w * E + e];
            smem[w * E + e] = run;
            run += v;
        }
        tb[e] = run;
    }
    __syncthreads();
    int32_t *sm = a.slot_map + (size_t)s * A;
#pragma unroll
    for (int r = 0; r < kHistRounds; ++r) {
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
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t *col = a.tile_base + (size_t)s * g.tiles * E + e;
        int run = 0;
        for (int t2 = 0; t2 < g.tiles; ++t2) {
            const int v = __ldcg(col + (size_t)t2 * E);
            __stcg(col + (size_t)t2 * E, run);
            run += v;
        }
        tot[e] = run;
        a.sp.send_counts[(size_t)s * E + e] = run;
        const int d = e / g.epr, le = e - d * g.epr;
        a.sp.recv_expert_counts[((size_t)d * R + s) * g.epr + le] = run;
    }
    __syncthreads();
    block_exclusive_scan(tot, E, wtot);
    for (int e = tid; e < E; e += blockDim.x) a.sp.send_offsets[(size_t)s * E + e] = tot[e];
    if (tid == 0) a.counters[s] = 0;  // re-arm for the next call

    // ---- last rank: cross-rank splits and window bases ------------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&a.counters[R], 1u) == (uint32_t)(R - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();

    int *rc = smem;              // [R][R] recv counts, destination-major
    int *ro = smem + R * R;      // [R][R] recv offsets
    int *wb = smem + 2 * R * R;  // [R]
    const int32_t *sc = a.sp.send_counts;
    const int32_t *so = a.sp.send_offsets;
    for (int p = tid; p < R * R; p += blockDim.x) {
        const int d = p / R, src = p - d * R;
        int c = 0;
        for (int le = 0; le < g.epr; ++le) c += __ldcg(sc + (size_t)src * E + d * g.epr + le);
        rc[p] = c;
        a.sp.recv_counts[p] = c;
    }
    __syncthreads();
    for (int d = tid; d < R; d += blockDim.x) {
        int run = 0;
        for (int src = 0; src < R; ++src) {
            ro[d * R + src] = run;
            a.sp.recv_offsets[d * R + src] = run;
            run += rc[d * R + src];
        }
        a.sp.recv_total[d] = run;
        wb[d] = run;
    }
    __syncthreads();
    if (tid == 0) {
        long long base = 0;
        bool ovf = false;
        for (int d = 0; d < R; ++d) {
            const int total_d = wb[d];
            const long long b = g.window_mode == A2AV_WINDOW_FIXED ? (long long)d * g.window_rows : base;
            if (g.window_mode == A2AV_WINDOW_FIXED && total_d > g.window_rows) ovf = true;
            a.sp.window_base[d] = (int32_t)b;
            base += total_d;
        }
        if (ovf) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
        a.counters[R] = 0;  // re-arm
    }
    for (int p = tid; p < R * E; p += blockDim.x) {
        const int src = p / E, e = p - src * E, d = e / g.epr;
        a.dest_base[p] = ro[d * R + src] + __ldcg(so + p) - __ldcg(so + (size_t)src * E + d * g.epr);
    }
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// ---------------------------------------------------------------------------
// Cluster splits kernel (R <= 16): one CTA per rank, all R CTAs in one
// thread-block cluster.  CTA s counts rank s (warp-aggregated, as above) and
// scans its counts in shared memory; after a cluster barrier every CTA reads
// the other ranks' send offsets straight out of their shared memory
// (distributed shared memory), derives the received counts, receive offsets
// and window bases, and writes the final arena row of each of its own
// assignments into slot_map.  No global atomics, fences or waits on other
// CTAs beyond the hardware cluster barrier.
// ---------------------------------------------------------------------------
constexpr int kClusterWarps = 32;
constexpr int kClusterThreads = kClusterWarps * 32;
constexpr int kClusterRounds = 8;  // rounds of 32 assignments per warp
constexpr int kClusterMaxRanks = 16;

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ const int *peer_smem(const int *p, int rank) {
    uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return reinterpret_cast<const int *>(static_cast<uintptr_t>(remote));
}
__device__ __forceinline__ int ld_dsmem(const int *p_cluster) {
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(v)
                 : "r"(static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p_cluster)))
                 : "memory");
    return v;
}

__global__ void __launch_bounds__(kClusterThreads, 1) splits_cluster_kernel(const HistArgs a) {
    extern __shared__ int smem[];
    grid_launch_dependents();
    const Geometry &g = a.g;
    const int R = g.R, E = g.E, epr = g.epr;
    const int A = g.T * g.k;
    const int s = blockIdx.x;  // == rank of this CTA in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = ((A + kClusterWarps - 1) / kClusterWarps + 31) / 32 * 32;
    const int a0 = warp * chunk;
    int *cnt = smem;                         // [32][E] per-warp counts -> warp bases
    int *so = cnt + kClusterWarps * E;       // [E + 1] send offsets of this rank (so[E] = total)
    int *rc = so + (E + 1);                  // [R][R] recv counts, [d][src]
    int *ro = rc + R * R;                    // [R] recv offsets of this rank in each window d
    int *wb = ro + R;                        // [R] window bases
    int *wtot = wb + R;                      // [33] scan scratch
    for (int i = tid; i < kClusterWarps * E; i += kClusterThreads) cnt[i] = 0;
    __syncthreads();

    int key[kClusterRounds], rank[kClusterRounds];
    bool bad = false;
    {
        const int32_t *idx = a.idx + (size_t)s * A;
        int *mine = cnt + warp * E;
        int vals[kClusterRounds];
#pragma unroll
        for (int r = 0; r < kClusterRounds; ++r) {
            const int ai = a0 + r * 32 + lane;
            vals[r] = (r * 32 < chunk && ai < A) ? __ldg(idx + ai) : -1;
        }
#pragma unroll
        for (int r = 0; r < kClusterRounds; ++r) {
            const int ai = a0 + r * 32 + lane;
            const bool inr = r * 32 < chunk && ai < A;
            const int e = vals[r];
            const bool good = inr && e >= 0 && e < E;
            bad |= inr && !good;
            const uint32_t peers = peers_by_ballot(good ? (uint32_t)e : (uint32_t)E, g.key_bits);
            const int before = __popc(peers & lanemask_lt());
            const int c = good ? mine[e] : 0;
            __syncwarp();
            if (good && before == 0) mine[e] = c + __popc(peers);
            __syncwarp();
            key[r] = good ? e : -1;
            rank[r] = c + before;
        }
        if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_BAD_EXPERT);
    }
    __syncthreads();

    // per expert: warp bases in warp order and the rank's totals
    for (int e = tid; e < E; e += kClusterThreads) {
        int run = 0;
        for (int w2 = 0; w2 < kClusterWarps; ++w2) {
            const int v = cnt[w2 * E + e];
            cnt[w2 * E + e] = run;
            run += v;
        }
        so[e] = run;
        a.sp.send_counts[(size_t)s * E + e] = run;
        const int d = e / epr, le = e - d * epr;
        a.sp.recv_expert_counts[((size_t)d * R + s) * epr + le] = run;
    }
    __syncthreads();
    const int total = block_exclusive_scan(so, E, wtot);
    if (tid == 0) so[E] = total;
    for (int e = tid; e < E; e += kClusterThreads) a.sp.send_offsets[(size_t)s * E + e] = so[e];
    __syncthreads();

    // every rank's send offsets are now in its CTA's shared memory
    cluster_barrier();
    for (int p = tid; p < R * R; p += kClusterThreads) {
        const int d = p / R, src = p - d * R;
        const int *pso = peer_smem(so, src);
        rc[p] = ld_dsmem(pso + (d + 1) * epr) - ld_dsmem(pso + d * epr);
    }
    __syncthreads();
    // no CTA may leave (its shared memory) until every peer has read it
    cluster_barrier();
    if (warp == 0) {
        // receive offsets of this rank in each window d, window totals and bases
        for (int d = 0; d < R; ++d) {
            const int v = lane < R ? rc[d * R + lane] : 0;
            const int incl = warp_inclusive_scan(v, lane);
            if (lane == s) ro[d] = incl - v;
            if (lane < R) {
                if (s == 0) a.sp.recv_offsets[d * R + lane] = incl - v;
                if (lane == s) a.sp.recv_counts[d * R + s] = v;
            }
            const int tot_d = __shfl_sync(kFull, incl, 31);
            if (lane == 0) wb[d] = tot_d;
        }
        __syncwarp();
        const int v = lane < R ? wb[lane] : 0;
        const int incl = warp_inclusive_scan(v, lane);
        const bool fixed = g.window_mode == A2AV_WINDOW_FIXED;
        const long long base = fixed ? (long long)lane * g.window_rows : (long long)(incl - v);
        const bool ovf = fixed && lane < R && v > g.window_rows;
        if (s == 0 && __any_sync(kFull, ovf) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
        __syncwarp();
        if (lane < R) {
            wb[lane] = (int)base;
            if (s == 0) {
                a.sp.window_base[lane] = (int)base;
                a.sp.recv_total[lane] = v;
            }
        }
    }
    __syncthreads();

    bool ovf = false;
    const int *mine = cnt + warp * E;
    int32_t *sm = a.slot_map + (size_t)s * A;
#pragma unroll
    for (int r = 0; r < kClusterRounds; ++r) {
        const int ai = a0 + r * 32 + lane;
        if (r * 32 < chunk && ai < A) {
            int32_t row = -1;
            const int e = key[r];
            if (e >= 0) {
                const int d = e / epr;
                const long long rel = (long long)ro[d] + so[e] - so[d * epr] + mine[e] + rank[r];
                if (g.window_mode == A2AV_WINDOW_FIXED && rel >= g.window_rows)
                    ovf = true;
                else
                    row = (int32_t)(wb[d] + rel);
            }
            sm[ai] = row;
        }
    }
    if (__any_sync(kFull, ovf) && lane == 0) atomicOr(a.status, (uint32_t)A2AV_DEV_WINDOW_OVERFLOW);
}

size_t cluster_smem_bytes(const Geometry &g) {
    return sizeof(int) * ((size_t)kClusterWarps * g.E + (g.E + 1) + (size_t)g.R * g.R + 2 * (size_t)g.R + 33);
}

bool cluster_eligible(const Geometry &g) {
    if (g.R > kClusterMaxRanks) return false;
    const long long A = (long long)g.T * g.k;
    const long long chunk = ((A + kClusterWarps - 1) / kClusterWarps + 31) / 32 * 32;
    return chunk <= 32 * kClusterRounds && cluster_smem_bytes(g) <= 160 * 1024;
}

size_t hist_smem_bytes(const Geometry &g) {
    const size_t a = (size_t)kHistWarps * g.E, b = 2 * (size_t)g.R * g.R + g.R;
    return sizeof(int) * (a > b ? a : b);
}

}  // namespace

cudaError_t configure_hist(a2av_plan_s &p) {
    if (!(p.cfg.flags & A2AV_FLAG_SPLITS_TILED) && cluster_eligible(p.g)) {
        cudaError_t e = cudaFuncSetAttribute(splits_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             160 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(splits_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        // Can a cluster of R such CTAs be resident at all on this device?
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(p.g.R);
        lc.blockDim = dim3(kClusterThreads);
        lc.dynamicSmemBytes = cluster_smem_bytes(p.g);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = p.g.R;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, splits_cluster_kernel, &lc);
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
    p.hist.smem = hist_smem_bytes(p.g);
    p.hist.grid = p.g.tiles;
    // Per-kernel cap shared by every plan: the largest any valid plan needs.
    Geometry worst{};
    worst.R = kMaxRanks;
    worst.E = kMaxExperts;
    return cudaFuncSetAttribute(hist_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)hist_smem_bytes(worst));
}

cudaError_t launch_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s) {
    if (p.splits_small) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(p.g.R);
        lc.blockDim = dim3(kClusterThreads);
        lc.dynamicSmemBytes = p.hist.smem;
        lc.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = p.g.R;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&lc, splits_cluster_kernel, a);
        if (e != cudaSuccess) return e;
    } else {
        dim3 grid(p.g.tiles, p.g.R);
        hist_scan_kernel<<<grid, p.hist.block, p.hist.smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace a2av
