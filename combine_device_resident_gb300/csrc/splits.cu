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
//     the same expert are grouped with __match_any_sync, so each group does
//     one shared-memory update (warp-aggregated counts) and each lane gets its
//     stable rank inside the warp's slice;
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
        const uint32_t peers = __match_any_sync(kFull, kk);
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

size_t hist_smem_bytes(const Geometry &g) {
    const size_t a = (size_t)kHistWarps * g.E, b = 2 * (size_t)g.R * g.R + g.R;
    return sizeof(int) * (a > b ? a : b);
}

}  // namespace

cudaError_t configure_hist(a2av_plan_s &p) {
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
    dim3 grid(p.g.tiles, p.g.R);
    hist_scan_kernel<<<grid, p.hist.block, p.hist.smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace a2av
