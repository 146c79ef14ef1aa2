// Internal declarations shared by the library's translation units: the plan,
// the kernel argument blocks, the launchers, and small PTX helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "a2av.h"

namespace a2av {

// Histogram tile: WARPS warps x ROUNDS rounds of 32 assignments.
constexpr int kHistWarps = 8;
constexpr int kHistRounds = 8;
constexpr int kHistThreads = kHistWarps * 32;
constexpr int kHistTile = kHistThreads * kHistRounds;  // assignments per tile

constexpr int kMaxRanks = 64;
constexpr int kMaxExperts = 2048;
constexpr int kMaxTopk = 32;

// Status bit set when a bounded wait gives up (should never happen: every wait
// in these kernels is on copies this CTA issued itself).
constexpr uint32_t kDevWaitTimeout = 1u << 31;

struct Splits {
    int32_t *send_counts, *send_offsets, *recv_counts, *recv_offsets, *recv_expert_counts, *recv_total,
        *window_base;
};

// Geometry every kernel needs.
struct Geometry {
    int32_t R, E, T, H, k, epr;
    int32_t tiles;        // histogram tiles per rank
    int32_t window_mode;  // 0 packed, 1 fixed
    int64_t window_rows;
};

struct HistArgs {
    Geometry g;
    const int32_t *idx;
    int32_t *slot_map;   // receives the rank of each assignment inside its tile
    int32_t *tile_base;  // [R][tiles][E] counts, turned into exclusive bases
    int32_t *dest_base;  // [R][E] window-relative first row of (source, expert)
    uint32_t *counters;  // [R + 1] last-block-done counters (left at 0)
    uint32_t *status;
    Splits sp;
};

struct PackArgs {
    Geometry g;
    const uint16_t *x;
    const int32_t *idx;
    int32_t *slot_map;
    const int32_t *tile_base;
    const int32_t *dest_base;
    const int32_t *window_base;
    uint16_t *recv;
    uint32_t *status;
    // TMA variant: chunking of a row into stage-sized pieces
    int32_t chunk_bytes;  // bytes per stage buffer (multiple of 16)
    int32_t nchunks;      // chunks per row
    int32_t stages;
};

struct CombineArgs {
    Geometry g;
    const uint16_t *y;
    const float *gate;
    const int32_t *slot_map;
    uint16_t *out;
    int64_t arena_rows;  // rows of y; a slot outside [0, arena_rows) is skipped and flagged
    uint32_t *status;
};

struct ScaleArgs {
    Geometry g;
    const uint16_t *recv;
    const int32_t *idx;
    const int32_t *slot_map;
    uint16_t *y;
    int64_t arena_rows;
    uint32_t *status;
};

// Status bit for a slot_map entry outside the arena handed to combine or the
// expert stand-in (the row is skipped, nothing is read or written there).
constexpr uint32_t kDevBadSlot = 1u << 2;

// Launch geometry chosen once per plan.
struct LaunchShape {
    int grid = 0;
    int block = 0;
    size_t smem = 0;
};

}  // namespace a2av

struct a2av_plan_s {
    a2av_config_t cfg;
    a2av::Geometry g;
    int num_sms = 0;
    void *workspace = nullptr;  // one device allocation
    size_t workspace_bytes = 0;
    int32_t *tile_base = nullptr;
    int32_t *dest_base = nullptr;
    uint32_t *counters = nullptr;
    uint32_t *status = nullptr;
    a2av::LaunchShape hist, pack, combine, scale;
    int pack_tma = 1;
    int32_t pack_chunk_bytes = 0, pack_nchunks = 0, pack_stages = 0;
    int64_t launches = 0;
};

namespace a2av {

// Launchers (return the cudaGetLastError() after the launch).
cudaError_t launch_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s);
cudaError_t launch_pack(const a2av_plan_s &p, const PackArgs &a, cudaStream_t s);
cudaError_t launch_combine(const a2av_plan_s &p, const CombineArgs &a, cudaStream_t s);
cudaError_t launch_scale(const a2av_plan_s &p, const ScaleArgs &a, cudaStream_t s);

// Records the text a2av_last_error() returns on the calling thread.
void set_last_error(const char *msg);

// Plan-time configuration of each kernel (attributes, occupancy, grid).
cudaError_t configure_hist(a2av_plan_s &p);
cudaError_t configure_pack(a2av_plan_s &p);
cudaError_t configure_combine(a2av_plan_s &p);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 16-byte streaming load of data that is read once and not written by the kernel.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream_v4(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace a2av
