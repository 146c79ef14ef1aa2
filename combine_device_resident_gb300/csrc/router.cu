// The router in front of the dispatch: per token, the k experts with the
// largest logits and the softmax of those logits as gate weights.  (NCCLX
// pages: abhik.ai, section on inference, Figure 13 -- a router chooses each
// token's experts; the pages do not define it, this is the plain
// top-k-then-softmax reading, with the tie, NaN and signed-zero rules of
// route_select.cuh.)
//
// Two kernels, the plan picks one (A2AV_FLAG_ROUTE_WARP: always the second).
//
// Lane kernel (E a multiple of 4, k <= 8, rows that fit shared memory; the
// default): P lanes per token (4; 2 for k = 2), 32/P tokens per warp task,
// four independent warps per CTA.  A task's logit rows come into shared
// memory by one bulk copy each, padded so that the 8 lanes of a quarter warp
// read 8 distinct bank groups; lane share r of a token holds 16-byte units
// r, r+P, ... of its row.  Per share, in three passes over it:
//   1. a lower bound tau of the k-th largest logit: the KMAX-th largest of
//      2*KMAX group maxima of the row, 2*KMAX/P of them per share, found by
//      merging the shares' sorted maxima over shuffles -- KMAX >= k distinct
//      elements are >= tau.  (For k = 1, P > KMAX: the row's maximum.)
//   2. a bit per logit of the share: set where the logit is >= tau (on
//      Gaussian logits with E = 256, k = 8: 10.4 per token, 2.6 per share,
//      at most 6 in a warp on average; a bound from each share's own maxima
//      let 16 per token through, and the minimum of KMAX group maxima 21);
//   3. a sorted insertion of the candidates, taken in ascending id order
//      from the bits, into KMAX registers, where only a strictly greater key
//      moves up (of equal logits the lower id, which arrived first, stays
//      ahead).
// A share whose tau is -infinity (a group of only -infinity or NaN logits)
// inserts every logit it holds instead.  Bitonic merges over xor shuffles
// then give every lane of the token the token's best KMAX, by key and then
// lower id.  Gates are computed as in route_token, so the two kernels give
// the same bits.
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

// Sort a bitonic sequence of floats in descending order (half-cleaners).
template <int L>
__device__ __forceinline__ void bitonic_desc(float (&v)[L]) {
#pragma unroll
    for (int d = L / 2; d >= 1; d >>= 1)
#pragma unroll
        for (int j = 0; j < L; ++j)
            if ((j & d) == 0) {
                const float hi = fmaxf(v[j], v[j + d]), lo = fminf(v[j], v[j + d]);
                v[j] = hi;
                v[j + d] = lo;
            }
}

// The K-th largest of the 2K values held by the P lanes of a token, each
// lane holding 2K/P of them sorted in descending order (P = 2 or 4).  The
// last step uses that of two sorted lists A and B of K, the K-th largest of
// both is min_i max(A_i, B_{K-1-i}).
template <int K, int P>
__device__ __forceinline__ float token_kth(float (&g)[2 * K / P]) {
    if constexpr (P == 2) {
        float t = INFINITY;
#pragma unroll
        for (int i = 0; i < K; ++i) t = fminf(t, fmaxf(g[i], __shfl_xor_sync(kAllLanes, g[K - 1 - i], 1)));
        return t;
    } else {
        constexpr int L = 2 * K / P;  // K / 2
        float c[2 * L];               // this pair's values, sorted: mine then the partner's reversed
#pragma unroll
        for (int i = 0; i < L; ++i) {
            c[i] = g[i];
            c[2 * L - 1 - i] = __shfl_xor_sync(kAllLanes, g[i], 1);
        }
        bitonic_desc<2 * L>(c);
        float t = INFINITY;
#pragma unroll
        for (int i = 0; i < K; ++i) t = fminf(t, fmaxf(c[i], __shfl_xor_sync(kAllLanes, c[K - 1 - i], 2)));
        return t;
    }
}

// Composite order of the selection: a larger key first, of equal keys the
// lower id.
__device__ __forceinline__ bool ranks_before(uint32_t ka, int ia, uint32_t kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Merge this lane's sorted list with that of lane ^ mask, keeping the best
// KMAX in order; both lanes end with the same list.  The better of a[j] and
// b[KMAX-1-j] for every j are the best KMAX of the two (a bitonic
// sequence); half-cleaners then sort them.
template <int KMAX>
__device__ __forceinline__ void merge_lists(uint32_t (&kk)[KMAX], int (&ii)[KMAX], int mask) {
    uint32_t bk[KMAX];
    int bi[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        bk[j] = __shfl_xor_sync(kAllLanes, kk[j], mask);
        bi[j] = __shfl_xor_sync(kAllLanes, ii[j], mask);
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const uint32_t ok = bk[KMAX - 1 - j];
        const int oi = bi[KMAX - 1 - j];
        if (!ranks_before(kk[j], ii[j], ok, oi)) {
            kk[j] = ok;
            ii[j] = oi;
        }
    }
#pragma unroll
    for (int d = KMAX / 2; d >= 1; d >>= 1)
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if ((j & d) == 0 && ranks_before(kk[j + d], ii[j + d], kk[j], ii[j])) {
                const uint32_t tk = kk[j];
                const int ti = ii[j];
                kk[j] = kk[j + d];
                ii[j] = ii[j + d];
                kk[j + d] = tk;
                ii[j + d] = ti;
            }
}

// Lanes per token: KMAX >= P lets every lane bound its share with its own
// group maxima (k = 1 takes the maximum over the token's lanes instead).
__host__ __device__ constexpr int lanes_per_token(int kmax) { return kmax >= 4 ? 4 : kmax == 2 ? 2 : 4; }
constexpr int kRouteWarps = 4;  // warps per CTA, each on its own tasks and shared memory

// Row stride in 16-byte units: at least E/4 and congruent to P mod 2P, so
// the 8 lanes of a quarter warp (8/P tokens, P lanes each on consecutive
// units of its row) read 8 distinct bank groups.
int lane_row_units(int E, int P) {
    int S = E / 4;
    while (S % (2 * P) != P) ++S;
    return S;
}
// One warp's shared memory: 32/P rows and the barrier.
size_t lane_warp_bytes(int E, int P) { return (size_t)(32 / P) * lane_row_units(E, P) * 16 + 16; }

// Mask words per lane share: its logits (4 per 16-byte unit, units r, r+P,
// ...) as bits, rounded up to 1, 2, 4 or 8 words; 0 when more are needed.
int lane_mask_words(int E, int P) {
    const int per = 4 * ((E / 4 + P - 1) / P);
    const int w = (per + 31) / 32;
    return w <= 1 ? 1 : w <= 2 ? 2 : w <= 4 ? 4 : w <= 8 ? 8 : 0;
}

// m[w] with a run-time w, by selects (a register array indexed at run time
// would go to local memory).
template <int MW>
__device__ __forceinline__ uint32_t pick_word(const uint32_t (&m)[MW], int w) {
    uint32_t v = m[0];
#pragma unroll
    for (int q = 1; q < MW; ++q)
        if (w == q) v = m[q];
    return v;
}

template <int KMAX, int MW>
__global__ void __launch_bounds__(32 * kRouteWarps) route_lane_kernel(const RouteArgs a) {
    constexpr int P = lanes_per_token(KMAX);
    constexpr int TPW = 32 / P;  // tokens per warp task
    extern __shared__ __align__(16) unsigned char sm[];
    const Geometry &g = a.g;
    const int E = g.E, k = g.k, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S4 = a.rsw;  // row stride in floats
    const size_t wbytes = (size_t)TPW * S4 * 4 + 16;
    unsigned char *base = sm + warp * wbytes;
    float *stage = reinterpret_cast<float *>(base);  // [TPW][S4]
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + wbytes - 16);
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int t = lane / P, r = lane - t * P;  // this lane: token t of the task, share r of its row
    const float4 *row4 = reinterpret_cast<const float4 *>(stage + (size_t)t * S4);
    const float *row = stage + (size_t)t * S4;
    const int nu = E / 4;
    const uint32_t rowb = (uint32_t)E * 4;
    const int ntok = g.R * g.T;
    const int ntask = (ntok + TPW - 1) / TPW;
    uint32_t phase = 0;
    for (int task = blockIdx.x * kRouteWarps + warp; task < ntask; task += gridDim.x * kRouteWarps) {
        const int u = task * TPW + t;
        bool act = u < ntok;
        if (act) {
            const int s = u / g.T;
            act = u - s * g.T < active_tokens(a.num_tokens, s, g.T);
        }
        const uint32_t lead = __ballot_sync(kAllLanes, act && r == 0);  // one copy per active token
        if (!lead) continue;
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(lead) * rowb);
        __syncwarp();
        if (act && r == 0) bulk_load(stage + (size_t)t * S4, a.logits + (size_t)u * E, rowb, bar);
        if (!__all_sync(kAllLanes, mbar_wait_bounded(bar, phase, a.wait_polls))) {
            // give up: let this warp's copies land (full bound), flag, leave
            mbar_wait_bounded(bar, phase, kWaitLimit);
            if (lane == 0) atomicOr(a.status, kDevWaitTimeout);
            return;
        }
        phase ^= 1;

        // 1. the bound.  Lane share r holds units r, r+P, ... of the row.
        float tau;
        if constexpr (KMAX >= P) {
            // the KMAX-th largest of the token's 2*KMAX group maxima, 2*KMAX/P
            // of them per share (NaN ignored by fmaxf; an all-NaN group stays
            // -infinity): KMAX distinct elements are >= tau
            constexpr int RK = KMAX / P, GL = 2 * RK;
            float gm[GL];
#pragma unroll
            for (int q = 0; q < GL; ++q) gm[q] = -INFINITY;
            for (int j0 = r; j0 < nu; j0 += P * GL) {
#pragma unroll
                for (int q = 0; q < GL; ++q) {
                    const int j = j0 + P * q;
                    if (j < nu) {
                        const float4 v = row4[j];
                        gm[q] = fmaxf(gm[q], fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                    }
                }
            }
            sort_desc<GL>(gm);
            tau = token_kth<KMAX, P>(gm);
        } else {
            // k = 1: the row's maximum
            tau = -INFINITY;
            for (int j = r; j < nu; j += P) {
                const float4 v = row4[j];
                tau = fmaxf(tau, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            }
#pragma unroll
            for (int m = 1; m < P; m <<= 1) tau = fmaxf(tau, __shfl_xor_sync(kAllLanes, tau, m));
        }

        // 2. this share's candidates, as bits: logit i of the share (unit
        // r + P*(i/4), lane i%4 of it) >= tau sets bit i (NaN never does;
        // with tau = -infinity the share is scanned whole below)
        uint32_t msk[MW];
        int cnt = 0;
#pragma unroll
        for (int w = 0; w < MW; ++w) {
            uint32_t bits = 0;
#pragma unroll
            for (int m8 = 0; m8 < 8; ++m8) {
                const int j = r + P * (w * 8 + m8);
                if (j < nu) {
                    const float4 v = row4[j];
                    bits |= ((uint32_t)(v.x >= tau) | (uint32_t)(v.y >= tau) << 1 | (uint32_t)(v.z >= tau) << 2 |
                             (uint32_t)(v.w >= tau) << 3)
                            << (4 * m8);
                }
            }
            msk[w] = bits;
            cnt += __popc(bits);
        }
        const bool scan_all = act && tau == -INFINITY;

        // 3. sorted insertion of the share's candidates, ascending ids: the
        // set bits in order, a cursor stepping through the words
        uint32_t kk[KMAX];
        int ii[KMAX];
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            kk[q] = 0u;
            ii[q] = -1;
        }
        const int nc = act && !scan_all ? cnt : 0;
        const int mc = (int)__reduce_max_sync(kAllLanes, (uint32_t)nc);
        int cw = 0;
        uint32_t cur = msk[0];
        for (int m = 0; m < mc; ++m) {
            uint32_t xk = 0u;
            int xi = 0;
            if (m < nc) {
                while (cur == 0 && cw < MW - 1) cur = pick_word<MW>(msk, ++cw);  // m < nc: bits are left
                if (cur) {
                    const int i = cw * 32 + __ffs(cur) - 1;
                    cur &= cur - 1;
                    xi = 4 * (r + P * (i >> 2)) + (i & 3);
                    xk = order_key(logit_key(row[xi]));
                }
            }
            insert_sorted<KMAX>(kk, ii, xk, xi);
        }
        if (__any_sync(kAllLanes, scan_all))
            for (int j = r; j < nu; j += P) {
                const float4 v = row4[j];
                const int e = 4 * j;
                insert_sorted<KMAX>(kk, ii, scan_all ? order_key(logit_key(v.x)) : 0u, e);
                insert_sorted<KMAX>(kk, ii, scan_all ? order_key(logit_key(v.y)) : 0u, e + 1);
                insert_sorted<KMAX>(kk, ii, scan_all ? order_key(logit_key(v.z)) : 0u, e + 2);
                insert_sorted<KMAX>(kk, ii, scan_all ? order_key(logit_key(v.w)) : 0u, e + 3);
            }
        // the token's P shares: every lane of it ends with the token's list
#pragma unroll
        for (int m = 1; m < P; m <<= 1) merge_lists<KMAX>(kk, ii, m);

        // Gates: softmax of the selected logits, summed in slot order.  Share
        // r computes and stores slots r, r+P, ...; the sum gathers every
        // slot's exponential from its share (all of a token's lanes see the
        // same list, so the same top and the same sum).
        {
            constexpr int SL = (KMAX + P - 1) / P;  // slots per share
            const float top = order_value(kk[0]);
            const bool flat = top == -INFINITY;      // every selected logit -infinity
            // this share's slots, picked with static indices (a register
            // array indexed by the lane's share would go to local memory)
            uint32_t sk[SL];
            int si[SL];
#pragma unroll
            for (int q = 0; q < SL; ++q) {
                sk[q] = 0u;
                si[q] = -1;
#pragma unroll
                for (int d = 0; d < P; ++d)
                    if (q * P + d < KMAX && d == r) {
                        sk[q] = kk[q * P + d];
                        si[q] = ii[q * P + d];
                    }
            }
            float ex[SL];
#pragma unroll
            for (int q = 0; q < SL; ++q) {
                const int j = q * P + r;
                ex[q] = (j < k && !flat) ? expf(order_value(sk[q]) - top) : 0.f;
            }
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const float ej = __shfl_sync(kAllLanes, ex[j / P], (lane & ~(P - 1)) | (j % P));
                if (j < k) sum = __fadd_rn(sum, ej);
            }
            if (act)
#pragma unroll
                for (int q = 0; q < SL; ++q) {
                    const int j = q * P + r;
                    if (j < k) {
                        a.idx[(size_t)u * k + j] = si[q];
                        a.gate[(size_t)u * k + j] = flat ? __fdiv_rn(1.0f, (float)k) : __fdiv_rn(ex[q], sum);
                    }
                }
        }
        __syncwarp();  // every lane is done with the rows before the next copies land
    }
}

template <int KMAX>
RouteKernel route_lane_kernel_mw(int mw) {
    switch (mw) {
        case 1: return route_lane_kernel<KMAX, 1>;
        case 2: return route_lane_kernel<KMAX, 2>;
        case 4: return route_lane_kernel<KMAX, 4>;
        case 8: return route_lane_kernel<KMAX, 8>;
        default: return nullptr;
    }
}
RouteKernel route_lane_kernel_for(int kmax, int mw) {
    switch (kmax) {
        case 1: return route_lane_kernel_mw<1>(mw);
        case 2: return route_lane_kernel_mw<2>(mw);
        case 4: return route_lane_kernel_mw<4>(mw);
        case 8: return route_lane_kernel_mw<8>(mw);
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
    if (kmax == 0 || E % 4 != 0 || E > 65535) return cudaSuccess;
    const int P = lanes_per_token(kmax);
    const size_t smem = kRouteWarps * lane_warp_bytes(E, P);
    const int mw = lane_mask_words(E, P);
    if (smem > kLaneSmemMax || mw == 0) return cudaSuccess;
    RouteKernel kern = route_lane_kernel_for(kmax, mw);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kRouteWarps, smem);
    if (e != cudaSuccess) return e;
    if (per_sm <= 0) return cudaSuccess;
    p.route_lane_kmax = kmax;
    p.route_lane_mw = mw;
    p.route_lane_rsw = 4 * lane_row_units(E, P);
    p.route_lane.grid = p.num_sms * per_sm;
    p.route_lane.block = 32 * kRouteWarps;
    p.route_lane.smem = smem;
    return cudaSuccess;
}

cudaError_t launch_route(const a2av_plan_s &p, const RouteArgs &a, cudaStream_t s) {
    // the lane kernel's row copies start on 16-byte boundaries: rows of E
    // floats with E % 4 == 0, from a 16-byte aligned logits array
    if (p.route_lane_kmax > 0 && reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) {
        RouteArgs b = a;
        b.rsw = p.route_lane_rsw;
        route_lane_kernel_for(p.route_lane_kmax, p.route_lane_mw)<<<p.route_lane.grid, p.route_lane.block,
                                                                      p.route_lane.smem, s>>>(b);
    } else {
        route_kernel_for(p.g.E)<<<p.route.grid, p.route.block, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace a2av
