// Combine: the return trip of the MoE exchange.  For every token the k expert
// outputs are gathered from the windows and summed with the gate weights:
//   out[s][t] = bf16_rne( sum_{j=0..k-1, slot>=0} w[s][t][j] * y[slot_map[s][t][j]] )
// accumulated in fp32 from 0 in slot order, with each product and each sum
// rounded on its own (__fmul_rn / __fadd_rn: no FMA contraction), so the
// result does not depend on the launch shape.  NCCLX pages: qiguanping deep
// dive section 7, Figure 13 (the dispatch shuffle and the combine).
//
// Warp per token; 16-byte vector gathers.  The kernel is instantiated for
// k in {1, 2, 4, 8} so that all k*U loads of a step are in flight before the
// ordered accumulation; other k use the generic loop.
//
// Also here: the expert stand-in of the checkable workload,
// y = bf16_rne(recv * (1 + e/E)), and its launcher.
#include <cuda_bf16.h>

#include "a2av_internal.cuh"

namespace a2av {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__device__ __forceinline__ void accumulate2(float &a0, float &a1, uint32_t q, float w) {
    a0 = __fadd_rn(a0, __fmul_rn(w, bf16lo(q)));
    a1 = __fadd_rn(a1, __fmul_rn(w, bf16hi(q)));
}

__device__ __forceinline__ void accumulate(float (&acc)[8], const uint4 &v, float w) {
    accumulate2(acc[0], acc[1], v.x, w);
    accumulate2(acc[2], acc[3], v.y, w);
    accumulate2(acc[4], acc[5], v.z, w);
    accumulate2(acc[6], acc[7], v.w, w);
}

__device__ __forceinline__ uint4 to_bf16x8(const float (&acc)[8]) {
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    return o;
}

template <int KT, int U>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
    const Geometry &g = a.g;
    const int k = KT > 0 ? KT : g.k;
    const int lane = threadIdx.x & 31;
    const long long ntok = (long long)g.R * g.T;
    const int nv = g.H >> 3;
    const size_t rowb = (size_t)g.H * 2;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    const char *y = reinterpret_cast<const char *>(a.y);
    bool bad_slot = false;
    for (long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < ntok; u += nw) {
        int32_t row = -1;
        float w = 0.f;
        if (lane < k) {
            row = __ldg(a.slot_map + (size_t)u * k + lane);
            w = __ldg(a.gate + (size_t)u * k + lane);
            if (row >= a.arena_rows) {
                bad_slot = true;
                row = -1;
            }
        }
        char *dst = reinterpret_cast<char *>(a.out) + (size_t)u * rowb;
        for (int vb = 0; vb < nv; vb += 32 * U) {
            float acc[U][8];
#pragma unroll
            for (int q = 0; q < U; ++q)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
            if constexpr (KT > 0) {
                uint4 buf[KT][U];
                int32_t rows[KT];
#pragma unroll
                for (int j = 0; j < KT; ++j)
#pragma unroll
                    for (int q = 0; q < U; ++q) buf[j][q] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int j = 0; j < KT; ++j) {
                    rows[j] = __shfl_sync(kFull, row, j);
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = vb + q * 32 + lane;
                        if (rows[j] >= 0 && v < nv) buf[j][q] = ld_stream_v4(y + (size_t)rows[j] * rowb + (size_t)v * 16);
                    }
                }
#pragma unroll
                for (int j = 0; j < KT; ++j) {
                    const float wj = __shfl_sync(kFull, w, j);
                    if (rows[j] < 0) continue;
#pragma unroll
                    for (int q = 0; q < U; ++q) accumulate(acc[q], buf[j][q], wj);
                }
            } else {
                for (int j = 0; j < k; ++j) {
                    const int32_t rj = __shfl_sync(kFull, row, j);
                    const float wj = __shfl_sync(kFull, w, j);
                    if (rj < 0) continue;
                    uint4 buf[U];
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = vb + q * 32 + lane;
                        buf[q] = make_uint4(0u, 0u, 0u, 0u);
                        if (v < nv) buf[q] = ld_stream_v4(y + (size_t)rj * rowb + (size_t)v * 16);
                    }
#pragma unroll
                    for (int q = 0; q < U; ++q) accumulate(acc[q], buf[q], wj);
                }
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int v = vb + q * 32 + lane;
                if (v < nv) st_stream_v4(dst + (size_t)v * 16, to_bf16x8(acc[q]));
            }
        }
    }
    if (__any_sync(kFull, bad_slot) && lane == 0) atomicOr(a.status, kDevBadSlot);
}

// y[row] = bf16_rne(float(recv[row]) * (1 + e/E)); y may alias recv (each row
// is owned by exactly one assignment, read and written by the same lane).
__global__ void __launch_bounds__(256) expert_scale_kernel(const ScaleArgs a) {
    const Geometry &g = a.g;
    const int lane = threadIdx.x & 31;
    const long long nass = (long long)g.R * g.T * g.k;
    const int nv = g.H >> 3;
    const size_t rowb = (size_t)g.H * 2;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long ga = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; ga < nass; ga += nw) {
        const int32_t row = a.slot_map[ga];
        if (row < 0) continue;
        if (row >= a.arena_rows) {
            if (lane == 0) atomicOr(a.status, kDevBadSlot);
            continue;
        }
        const int e = a.idx[ga];
        const float scale = __fadd_rn(1.0f, __fdiv_rn((float)e, (float)g.E));
        const char *src = reinterpret_cast<const char *>(a.recv) + (size_t)row * rowb;
        char *dst = reinterpret_cast<char *>(a.y) + (size_t)row * rowb;
        for (int v = lane; v < nv; v += 32) {
            const uint4 in = *reinterpret_cast<const uint4 *>(src + (size_t)v * 16);
            const uint32_t q[4] = {in.x, in.y, in.z, in.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = pack_bf16x2(__fmul_rn(bf16lo(q[i]), scale), __fmul_rn(bf16hi(q[i]), scale));
            *reinterpret_cast<uint4 *>(dst + (size_t)v * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

template <int KT, int U>
cudaError_t occupancy_grid(const a2av_plan_s &p, int &grid) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<KT, U>, 256, 0);
    grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    return e;
}

}  // namespace

cudaError_t configure_combine(a2av_plan_s &p) {
    p.combine.block = 256;
    p.scale.block = 256;
    cudaError_t e;
    switch (p.g.k) {
        case 1: e = occupancy_grid<1, 4>(p, p.combine.grid); break;
        case 2: e = occupancy_grid<2, 4>(p, p.combine.grid); break;
        case 4: e = occupancy_grid<4, 2>(p, p.combine.grid); break;
        case 8: e = occupancy_grid<8, 2>(p, p.combine.grid); break;
        default: e = occupancy_grid<0, 2>(p, p.combine.grid); break;
    }
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, expert_scale_kernel, 256, 0);
    p.scale.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    return e;
}

cudaError_t launch_combine(const a2av_plan_s &p, const CombineArgs &a, cudaStream_t s) {
    switch (p.g.k) {
        case 1: combine_kernel<1, 4><<<p.combine.grid, 256, 0, s>>>(a); break;
        case 2: combine_kernel<2, 4><<<p.combine.grid, 256, 0, s>>>(a); break;
        case 4: combine_kernel<4, 2><<<p.combine.grid, 256, 0, s>>>(a); break;
        case 8: combine_kernel<8, 2><<<p.combine.grid, 256, 0, s>>>(a); break;
        default: combine_kernel<0, 2><<<p.combine.grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_scale(const a2av_plan_s &p, const ScaleArgs &a, cudaStream_t s) {
    expert_scale_kernel<<<p.scale.grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace a2av
