// Per-token routing by one warp, shared by the router kernel and the
// histogram kernel that routes its own tile: the k largest of E logits, in
// descending order, equal logits by lower expert id, a NaN logit counted as
// -infinity and -0 as +0; gates = the softmax of the selected logits,
// exp(l_j - l_0) / sum_i exp(l_i - l_0) summed in slot order, or 1/k each if
// every selected logit is -infinity.  (NCCLX pages: abhik.ai, section on
// inference, Figure 13 -- a router chooses each token's experts; the pages
// do not define the router, this is the plain top-k-then-softmax reading.)
//
// Lane l keeps the logits of experts e = q*32 + l (q < EPL) in registers as
// order-preserving integer keys; round j of k is two warp reductions
// (redux.sync): the largest key, then the lowest expert id holding it.
#pragma once
#include <math.h>
#include <stdint.h>

namespace a2av {

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

// Route the token whose E logits start at `l` (k <= E, E <= 32*EPL).  All
// 32 lanes call it; lane j < k gets slot j's expert id and gate, the other
// lanes -1 and 0.
template <int EPL>
__device__ __forceinline__ void route_token(const float *l, int E, int k, int lane, int32_t &id_out,
                                            float &gate_out) {
    constexpr uint32_t kAll = 0xffffffffu;
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
        const uint32_t top = __reduce_max_sync(kAll, best);
        const uint32_t id = __reduce_min_sync(kAll, best == top ? (uint32_t)(bq * 32 + lane) : 0xffffffffu);
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
    const float top = __shfl_sync(kAll, my_v, 0);
    float w;
    if (top == -INFINITY) {
        w = __fdiv_rn(1.0f, (float)k);
    } else {
        const float ex = lane < k ? expf(my_v - top) : 0.f;
        float sum = 0.f;
        for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, __shfl_sync(kAll, ex, i));
        w = __fdiv_rn(ex, sum);
    }
    id_out = lane < k ? my_i : -1;
    gate_out = lane < k ? w : 0.f;
}

}  // namespace a2av
