// The router in front of the dispatch: per token, the k experts with the
// largest logits and the softmax of those logits as gate weights (the
// selection itself is route_token in route_select.cuh).  One warp per
// token, grid-stride over all R*T tokens; tokens past a rank's active count
// are skipped.
#include "a2av_internal.cuh"
#include "route_select.cuh"

namespace a2av {
namespace {

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
