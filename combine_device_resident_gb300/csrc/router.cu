// The router in front of the dispatch: per token, the k experts with the
// largest logits and the softmax of those logits as gate weights.  NCCLX
// pages: abhik.ai, section on inference, Figure 13 (a router chooses each
// token's experts before the tokens are sorted by expert).  The pages do not
// define the router; this one takes the k largest logits in descending
// order, equal logits by lower expert id, a NaN logit as -infinity, and the
// gates exp(l_j - l_0) / sum_i exp(l_i - l_0) summed in slot order (equal
// weights if every selected logit is -infinity).
//
// One warp per token.  Each lane loads its E/32 logits into registers once
// (as order-preserving integer keys); round j is two warp reductions
// (redux.sync): the largest key, then the lowest expert id holding it.
#include <math.h>

#include "a2av_internal.cuh"

namespace a2av {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

// NaN counts as -infinity; -0 as +0 (they compare equal, so the lower id wins).
__device__ __forceinline__ float logit_key(float v) { return v != v ? -INFINITY : (v == 0.0f ? 0.0f : v); }

// Order-preserving map of a (non-NaN) float to uint32: a > b as floats iff
// key(a) > key(b); -infinity maps to 0x007fffff, so 0 is below every logit.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// EPL = logits per lane held in registers (a power of two >= E/32).  Lane
// owns experts e = q*32 + lane, keeps their order keys, and zeroes a key
// once it is picked (or out of range).  A round is two warp reductions: the
// largest key, then the lowest expert id among the lanes holding it.
template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const RouteArgs a) {
    const Geometry &g = a.g;
    const int E = g.E, k = g.k, lane = threadIdx.x & 31;
    const long long ntok = (long long)g.R * g.T;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < ntok; u += nw) {
        const int s = (int)(u / g.T);
        if (u - (long long)s * g.T >= active_tokens(a.num_tokens, s, g.T)) continue;  // warp-uniform
        const float *l = a.logits + (size_t)u * E;
        uint32_t key[EPL];
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = q * 32 + lane;
            key[q] = e < E ? order_key(logit_key(__ldg(l + e))) : 0u;
        }
        float my_v = -INFINITY;
        int my_i = -1;
        for (int j = 0; j < k; ++j) {
            uint32_t best = 0u;
            int bq = 0;
#pragma unroll
            for (int q = 0; q < EPL; ++q)  // strict: the lower q (lower id) wins a tie
                if (key[q] > best) {
                    best = key[q];
                    bq = q;
                }
            const uint32_t top = __reduce_max_sync(kFull, best);
            const uint32_t id = __reduce_min_sync(kFull, best == top ? (uint32_t)(bq * 32 + lane) : 0xffffffffu);
            if ((int)(id & 31) == lane) {  // the owner retires the pick
#pragma unroll
                for (int q = 0; q < EPL; ++q)
                    if (q == (int)(id >> 5)) key[q] = 0u;
            }
            if (lane == j) {
                my_v = order_value(top);
                my_i = (int)id;
            }
        }
        const float top = __shfl_sync(kFull, my_v, 0);
        float w;
        if (top == -INFINITY) {
            w = __fdiv_rn(1.0f, (float)k);
        } else {
            const float ex = lane < k ? expf(my_v - top) : 0.f;
            float sum = 0.f;
            for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, __shfl_sync(kFull, ex, i));
            w = __fdiv_rn(ex, sum);
        }
        if (lane < k) {
            a.idx[(size_t)u * k + lane] = my_i;
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

}  // namespace

cudaError_t configure_route(a2av_plan_s &p) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_kernel_for(p.g.E), 256, 0);
    p.route.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    p.route.block = 256;
    return e;
}

cudaError_t launch_route(const a2av_plan_s &p, const RouteArgs &a, cudaStream_t s) {
    route_kernel_for(p.g.E)<<<p.route.grid, p.route.block, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace a2av
