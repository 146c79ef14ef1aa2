// The router in front of the dispatch: per token, the k experts with the
// largest logits and the softmax of those logits as gate weights.  (NCCLX
// pages: abhik.ai, section on inference, Figure 13 -- a router chooses each
// token's experts; the pages do not define it, this is the plain
// top-k-then-softmax reading, with the tie, NaN and signed-zero rules of
// route_select.cuh.)
//
// Two kernels, the plan picks one (A2AV_FLAG_ROUTE_WARP: always the second).
//
// Lane-per-token kernel (E a multiple of 4, k <= 8, rows that fit shared
// memory; the default): a warp takes 32 consecutive tokens and brings their
// logit rows into shared memory, one bulk copy per row, rows padded so that
// lane i reading row i with 16-byte loads touches distinct banks.  Each lane
// then selects its own token's k largest in three passes over its row:
//   1. the maxima of 2*KMAX disjoint groups of the row (16-byte unit j in
//      group j % (2*KMAX)), KMAX >= k.  tau, the KMAX-th largest of them,
//      bounds the k-th largest logit from below: the group maxima are
//      distinct elements, KMAX of them >= tau.  (Sort both halves of the
//      maxima; the KMAX-th largest of all is min_i max(A_i, B_{KMAX-1-i}),
//      the first step of a bitonic merge.)
//   2. the ids of the logits >= tau, in ascending id order, into the lane's
//      candidate list (about 10 per token on Gaussian logits with E = 256,
//      k = 8, at most 16 in a warp; with KMAX groups and their minimum it
//      was 21, and 8% of the lanes overflowed the list);
//   3. a sorted insertion of the candidates into KMAX registers, where only
//      a strictly greater key moves up: of equal logits the lower id stays
//      ahead, as it arrived first.
// A lane whose list overflows, or whose tau is -infinity (a group of only
// -infinity or NaN logits), inserts every logit of its row instead.  Gates
// are computed as in route_token, so both kernels give the same bits.
//
// Warp-per-token kernel (any shape): route_token in route_select.cuh, one
// warp per token, grid-stride over all R*T tokens.
//
// Tokens past a rank's active count are skipped by both.
#include "a2av_internal.cuh"
#include "route_select.cuh"

namespace a2av {
namespace {

constexpr uint32_t kAllLanes = 0xffffffffu;
constexpr int kLaneCap = 32;               // candidate list slots per lane (slot kLaneCap: overflow sink)
constexpr size_t kLaneSmemMax = 96 * 1024;  // rows bigger than this take the warp kernel

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const RouteArgs a) {
    const Geometry &g = a.g;
    const int E = g.E, k = g.k, lane = threadIdx.x & 31;
    // 32-bit token index (R*T < 2^31 for every valid plan): a 64-bit divide
    // here is a subroutine call, and the call pushed key[] out of registers
    // into the stack frame
    const int ntok = g.R * g.T;
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    for (int u = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); u < ntok; u += nw) {
        const int s = u / g.T;
        if (u - s * g.T >= active_tokens(a.num_tokens, s, g.T)) continue;  // warp-uniform
        int32_t id;
        float w;
        route_token<EPL>(a.logits + (size_t)u * E, E, k, lane, id, w);
        if (lane < k) {
            a.idx[(size_t)u * k + lane] = id;
            a.gate[(size_t)u * k + lane] = w;
        }
    }
}

using RouteKernel = void (*)(const RouteArgs);

RouteKernel route_kernel_for(int E) {
    const int need = (E + 31) / 32;
    if (need <= 1) return route_kernel<1>;
    if (need <= 2) return route_kernel<2>;
    if (need <= 4) return route_kernel<4>;
    if (need <= 8) return route_kernel<8>;
    if (need <= 16) return route_kernel<16>;
    if (need <= 32) return route_kernel<32>;
    return route_kernel<64>;
}

// Insert (xk, xi) into kk[0..KMAX) sorted by descending key.  A key of 0 is
// below every logit and never moves in.
template <int KMAX>
__device__ __forceinline__ void insert_sorted(uint32_t (&kk)[KMAX], int (&ii)[KMAX], uint32_t xk, int xi) {
    bool gt[KMAX];
#pragma unroll
    for (int p = 0; p < KMAX; ++p) gt[p] = xk > kk[p];
#pragma unroll
    for (int p = KMAX - 1; p > 0; --p) {  // descending p: kk[p - 1] still holds its old value
        kk[p] = gt[p - 1] ? kk[p - 1] : (gt[p] ? xk : kk[p]);
        ii[p] = gt[p - 1] ? ii[p - 1] : (gt[p] ? xi : ii[p]);
    }
    if (gt[0]) {
        kk[0] = xk;
        ii[0] = xi;
    }
}

// Sort n floats in descending order (a bubble network, no NaN inside).
template <int N>
__device__ __forceinline__ void sort_desc(float (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
        for (int j = 0; j + 1 < N - i; ++j) {
            const float hi = fmaxf(v[j], v[j + 1]), lo = fminf(v[j], v[j + 1]);
            v[j] = hi;
            v[j + 1] = lo;
        }
}

// Row stride in floats: a multiple of 4 with an odd number of 16-byte units,
// so lanes reading the same unit of their own rows hit distinct banks.
int lane_row_stride(int E) {
    const int u = E / 4;
    return 4 * (u + ((u & 1) ? 2 : 1));
}
size_t lane_smem_bytes(int E) {
    return (size_t)32 * lane_row_stride(E) * sizeof(float) + (size_t)(kLaneCap + 1) * 32 * sizeof(uint16_t) +
           sizeof(uint64_t);
}

template <int KMAX>
__global__ void __launch_bounds__(32) route_lane_kernel(const RouteArgs a) {
    extern __shared__ __align__(16) unsigned char sm[];
    const Geometry &g = a.g;
    const int E = g.E, k = g.k, lane = threadIdx.x, rsw = a.rsw;
    float *stage = reinterpret_cast<float *>(sm);                            // [32][rsw]
    uint16_t *lst = reinterpret_cast<uint16_t *>(stage + (size_t)32 * rsw);  // [kLaneCap + 1][32]
    uint64_t *bar = reinterpret_cast<uint64_t *>(lst + (kLaneCap + 1) * 32);
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const float *row = stage + (size_t)lane * rsw;
    const float4 *row4 = reinterpret_cast<const float4 *>(row);
    uint16_t *mine = lst + lane;
    const int nu = E / 4;
    const uint32_t rowb = (uint32_t)E * 4;
    const int ntok = g.R * g.T;
    const int ntask = (ntok + 31) / 32;
    uint32_t phase = 0;
    for (int task = blockIdx.x; task < ntask; task += gridDim.x) {
        const int u = task * 32 + lane;
        bool act = u < ntok;
        if (act) {
            const int s = u / g.T;
            act = u - s * g.T < active_tokens(a.num_tokens, s, g.T);
        }
        const uint32_t am = __ballot_sync(kAllLanes, act);
        if (!am) continue;
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(am) * rowb);
        __syncwarp();
        if (act) bulk_load(stage + (size_t)lane * rsw, a.logits + (size_t)u * E, rowb, bar);
        if (!__all_sync(kAllLanes, mbar_wait_bounded(bar, phase, a.wait_polls))) {
            // give up: let this CTA's copies land (full bound), flag, leave
            mbar_wait_bounded(bar, phase, kWaitLimit);
            if (lane == 0) atomicOr(a.status, kDevWaitTimeout);
            return;
        }
        phase ^= 1;

        // 1. maxima of 2*KMAX disjoint groups (NaN ignored: fmaxf returns the
        // other operand; a group of only NaN stays -infinity), then the
        // KMAX-th largest of them
        constexpr int G = 2 * KMAX;
        float ga[KMAX], gb[KMAX];
#pragma unroll
        for (int q = 0; q < KMAX; ++q) ga[q] = gb[q] = -INFINITY;
        for (int j0 = 0; j0 < nu; j0 += G) {
#pragma unroll
            for (int q = 0; q < G; ++q)
                if (j0 + q < nu) {
                    const float4 v = row4[j0 + q];
                    const float m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                    if (q < KMAX) ga[q] = fmaxf(ga[q], m);
                    else gb[q - KMAX] = fmaxf(gb[q - KMAX], m);
                }
        }
        sort_desc<KMAX>(ga);
        sort_desc<KMAX>(gb);
        float tau = fmaxf(ga[0], gb[KMAX - 1]);
#pragma unroll
        for (int i = 1; i < KMAX; ++i) tau = fminf(tau, fmaxf(ga[i], gb[KMAX - 1 - i]));

        // 2. candidates: ids of the logits >= tau, ascending (NaN never is;
        // with tau = -infinity the lane scans its whole row below instead)
        int cnt = 0;
#pragma unroll 4
        for (int j = 0; j < nu; ++j) {
            const float4 v = row4[j];
            const int e = 4 * j;
            if (v.x >= tau) mine[min(cnt++, kLaneCap) * 32] = (uint16_t)e;
            if (v.y >= tau) mine[min(cnt++, kLaneCap) * 32] = (uint16_t)(e + 1);
            if (v.z >= tau) mine[min(cnt++, kLaneCap) * 32] = (uint16_t)(e + 2);
            if (v.w >= tau) mine[min(cnt++, kLaneCap) * 32] = (uint16_t)(e + 3);
        }
        const bool scan_all = act && (tau == -INFINITY || cnt > kLaneCap);

        // 3. sorted insertion, candidates in ascending id order
        uint32_t kk[KMAX];
        int ii[KMAX];
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            kk[q] = 0u;
            ii[q] = -1;
        }
        const int nc = act && !scan_all ? cnt : 0;
        const int mc = (int)__reduce_max_sync(kAllLanes, (uint32_t)nc);
        for (int m = 0; m < mc; ++m) {
            uint32_t xk = 0u;
            int xi = 0;
            if (m < nc) {
                xi = mine[m * 32];
                xk = order_key(logit_key(row[xi]));
            }
            insert_sorted<KMAX>(kk, ii, xk, xi);
        }
        if (__any_sync(kAllLanes, scan_all))
            for (int e = 0; e < E; ++e) insert_sorted<KMAX>(kk, ii, scan_all ? order_key(logit_key(row[e])) : 0u, e);

        if (act) {
            // gates: softmax of the selected logits, summed in slot order
            const float top = order_value(kk[0]);
            float w[KMAX];
            if (top == -INFINITY) {
#pragma unroll
                for (int j = 0; j < KMAX; ++j) w[j] = __fdiv_rn(1.0f, (float)k);
            } else {
                float sum = 0.f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    w[j] = j < k ? expf(order_value(kk[j]) - top) : 0.f;
                    if (j < k) sum = __fadd_rn(sum, w[j]);
                }
#pragma unroll
                for (int j = 0; j < KMAX; ++j) w[j] = __fdiv_rn(w[j], sum);
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < k) {
                    a.idx[(size_t)u * k + j] = ii[j];
                    a.gate[(size_t)u * k + j] = w[j];
                }
        }
        __syncwarp();  // every lane is done with the rows before the next copies land
    }
}

RouteKernel route_lane_kernel_for(int kmax) {
    switch (kmax) {
        case 1: return route_lane_kernel<1>;
        case 2: return route_lane_kernel<2>;
        case 4: return route_lane_kernel<4>;
        case 8: return route_lane_kernel<8>;
        default: return nullptr;
    }
}

}  // namespace

cudaError_t configure_route(a2av_plan_s &p) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_kernel_for(p.g.E), 256, 0);
    if (e != cudaSuccess) return e;
    p.route.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    p.route.block = 256;
    p.route_lane_kmax = 0;
    if (p.cfg.flags & A2AV_FLAG_ROUTE_WARP) return cudaSuccess;
    const int k = p.g.k, E = p.g.E;
    const int kmax = k <= 1 ? 1 : k <= 2 ? 2 : k <= 4 ? 4 : k <= 8 ? 8 : 0;
    const size_t smem = lane_smem_bytes(E);
    if (kmax == 0 || E % 4 != 0 || E > 65535 || smem > kLaneSmemMax) return cudaSuccess;
    RouteKernel kern = route_lane_kernel_for(kmax);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm <= 0) return cudaSuccess;
    p.route_lane_kmax = kmax;
    p.route_lane_rsw = lane_row_stride(E);
    p.route_lane.grid = p.num_sms * per_sm;
    p.route_lane.block = 32;
    p.route_lane.smem = smem;
    return cudaSuccess;
}

cudaError_t launch_route(const a2av_plan_s &p, const RouteArgs &a, cudaStream_t s) {
    // the lane kernel's row copies start on 16-byte boundaries: rows of E
    // floats with E % 4 == 0, from a 16-byte aligned logits array
    if (p.route_lane_kmax > 0 && reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) {
        RouteArgs b = a;
        b.rsw = p.route_lane_rsw;
        route_lane_kernel_for(p.route_lane_kmax)<<<p.route_lane.grid, 32, p.route_lane.smem, s>>>(b);
    } else {
        route_kernel_for(p.g.E)<<<p.route.grid, p.route.block, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace a2av
