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
// Polls of a bounded mbarrier wait before it gives up (each poll is a
// try_wait, which itself blocks for a while): seconds, far beyond any copy.
constexpr long long kWaitLimit = 1ll << 22;

struct Splits {
    int32_t *send_counts, *send_offsets, *recv_counts, *recv_offsets, *recv_expert_counts, *recv_total,
        *window_base;
    int32_t *recv_expert_offsets;  // may be null in source order (then not written)
};

// Geometry every kernel needs.
struct Geometry {
    int32_t R, E, T, H, k, epr;
    int32_t key_bits;     // bits of an expert key in [0, E] (E marks a dropped id)
    int32_t tiles;        // histogram tiles per rank
    int32_t window_mode;  // A2AV_WINDOW_*
    int32_t recv_order;   // A2AV_ORDER_*
    int64_t window_rows;
};

struct HistArgs {
    Geometry g;
    const int32_t *num_tokens;  // [R] tokens taking part per rank, or null (all T)
    const int32_t *idx;
    int32_t *slot_map;   // receives the rank of each assignment inside its tile
    int32_t *tile_base;   // [R][tiles][E] counts, turned into exclusive bases
    int32_t *rank_total;  // [R] valid assignments of each source rank
    uint32_t *counters;   // [R + 1] last-block-done counters (left at 0)
    uint32_t *status;
    Splits sp;
    // routed variant (a2av_route_splits): logits in, topk_idx and gates out
    const float *logits;  // [R][T][E]
    int32_t *idx_out;     // [R][T][k]
    float *gate_out;      // [R][T][k]
};

struct PackArgs {
    Geometry g;
    const int32_t *num_tokens;
    const uint16_t *x;
    const int32_t *idx;
    int32_t *slot_map;
    const int32_t *tile_base;
    const int32_t *send_offsets;  // splits arrays written by the splits kernel
    const int32_t *recv_offsets;
    const int32_t *window_base;
    const int32_t *recv_expert_offsets;  // [R][R][Epr]; read in the expert-grouped order
    uint16_t *recv;
    uint32_t *status;
    // TMA variant: chunking of a row into stage-sized pieces
    int32_t chunk_bytes;  // bytes per stage buffer (multiple of 16)
    int32_t nchunks;      // chunks per row
    int32_t stages;
    int32_t rows_final;   // 1: slot_map already holds final rows (single-CTA splits)
    int32_t lag;          // store groups allowed to read a stage before it is refilled
    int64_t padded_tk;    // padded plans: T*k, and `recv` is the padded send buffer
    int32_t trigger_early;  // 1: let the dependent grid launch at once (few tokens: latency-bound call)
    int64_t wait_polls;     // main-loop mbarrier wait limit (kWaitLimit unless a2av_set_wait_limit)
};

struct RouteArgs {
    Geometry g;
    const int32_t *num_tokens;
    const float *logits;  // [R][T][E]
    int32_t *idx;         // [R][T][k]
    float *gate;          // [R][T][k]
    uint32_t *status;     // device status word (wait give-up bit)
    int64_t wait_polls;   // mbarrier wait limit of the lane-per-token kernel
    int32_t rsw;          // its padded shared-memory row stride, in floats
};

struct ExchangeArgs {
    const uint16_t *sendbuf;
    uint16_t *recv;
    int32_t R;
    int64_t block_vecs;  // 16-byte vectors per (source, destination) segment: T*k*H/8
};

struct CombineArgs {
    Geometry g;
    const int32_t *num_tokens;
    const uint16_t *y;
    const float *gate;
    const int32_t *slot_map;
    uint16_t *out;
    int64_t arena_rows;  // rows of y; a slot outside [0, arena_rows) is skipped and flagged
    uint32_t *status;
    // TMA variant
    int32_t chunk_bytes;  // bytes of a row per stage slot (multiple of 16)
    int32_t nchunks;      // chunks per row
    int32_t stages;
    int32_t nsplit;       // LSU variant: pieces per row
    int64_t wait_polls;   // TMA variant: main-loop mbarrier wait limit
    int32_t trigger_early;  // 1: let the next kernel (a programmatic dependent) launch at once (few tokens)
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
    int32_t *rank_total = nullptr;
    uint32_t *counters = nullptr;
    uint32_t *status = nullptr;
    a2av::LaunchShape hist, pack, combine, scale, exchange, route, route_lane;
    int splits_small = 0;  // 1: one-CTA splits kernel that writes final rows
    const int32_t *num_tokens = nullptr;  // a2av_set_active_tokens
    int combine_tma = 1;
    int32_t comb_chunk_bytes = 0, comb_nchunks = 0, comb_stages = 0, comb_nsplit = 1, comb_unroll = 2, comb_group = 1;
    bool comb_batch = false;  // combine_batched_kernel (set with few_tokens where rows split into pieces)
    bool few_tokens = false;  // R*T below the combine's warps: the pack triggers the combine's launch early
    int pack_tma = 1;
    int32_t pack_chunk_bytes = 0, pack_nchunks = 0, pack_stages = 0, pack_lag = 1;
    int pack_stream_rows = 0;  // the pack stores its rows evict-first (see configure_pack)
    int route_lane_kmax = 0;   // lane-per-token router instantiation (0: the warp-per-token kernel)
    int route_lane_mw = 0;     // its candidate mask words per lane share
    int32_t route_lane_rsw = 0;  // its padded row stride in floats
    int64_t launches = 0;
    int64_t wait_polls = a2av::kWaitLimit;  // main-loop wait limit of the TMA kernels (a2av_set_wait_limit)
    // 1: the last splits launch left final rows in slot_map (cluster kernel);
    // 0: tile ranks (tiled kernels).  The next pack reads it.
    int last_rows_final = 0;
};

namespace a2av {

// Launch with the programmatic stream-serialization attribute (the kernel
// calls grid_dependency_wait() before reading its predecessor's output).
template <typename Kernel, typename Args>
cudaError_t launch_pdl(Kernel kernel, int grid, int block, size_t smem, cudaStream_t s, const Args &args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

// Launchers (return the cudaGetLastError() after the launch).
cudaError_t launch_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s);
cudaError_t launch_pack(const a2av_plan_s &p, const PackArgs &a, cudaStream_t s);
cudaError_t launch_combine(const a2av_plan_s &p, const CombineArgs &a, cudaStream_t s);
cudaError_t launch_scale(const a2av_plan_s &p, const ScaleArgs &a, cudaStream_t s);
cudaError_t launch_exchange_padded(const a2av_plan_s &p, const ExchangeArgs &a, cudaStream_t s);
cudaError_t launch_route(const a2av_plan_s &p, const RouteArgs &a, cudaStream_t s);
// Router fused into the tiled histogram (E <= 256, k | 32); slot_map then
// holds tile ranks.
bool routed_splits_supported(const a2av_plan_s &p);
cudaError_t launch_routed_hist(const a2av_plan_s &p, const HistArgs &a, cudaStream_t s);
cudaError_t configure_route(a2av_plan_s &p);

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

// Lanes of the warp whose `key` equals this lane's, for keys in [0, 2^nbits):
// one ballot per key bit (a warp multisplit), all of them full-rate
// instructions.
__device__ __forceinline__ uint32_t peers_by_ballot(uint32_t key, int nbits) {
    uint32_t peers = 0xffffffffu;
    for (int b = 0; b < nbits; ++b) {
        const uint32_t bit = (key >> b) & 1u;
        const uint32_t set = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? set : ~set;
    }
    return peers;
}

// Tokens of rank s that take part in this call: all T, or the caller's
// device-resident count clamped to [0, T] (read when the kernel runs).
__device__ __forceinline__ int active_tokens(const int32_t *num_tokens, int s, int T) {
    if (!num_tokens) return T;
    const int n = __ldg(num_tokens + s);
    return n < 0 ? 0 : (n > T ? T : n);
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor runs; it
// must wait here before touching anything the predecessor writes.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the dependent grid begin launching (its wait still covers our writes).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bring the line holding p into L2 (no value is read; nothing waits on it).
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ void st_stream_v4(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA) helpers.  Every wait is bounded: a kernel that
// gives up sets a status bit and returns instead of hanging the GPU.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// At most `limit` polls (0: give up without polling).  Kernels take the
// main-loop limit from their arguments (a2av_set_wait_limit) and always
// drain their own copies with kWaitLimit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long limit = kWaitLimit) {
    for (long long it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// L2 policy: lines fetched with it are the first to be evicted.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// bulk_store with an L2 cache policy for the destination lines.
__device__ __forceinline__ void bulk_store_hint(void *dst, const void *src_smem, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_u32(src_smem)), "r"(bytes), "l"(policy)
                 : "memory");
}
// bulk_load with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_load_hint(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most `n` of this thread's newest bulk groups still read smem.
__device__ __forceinline__ void bulk_wait_read_upto(int n) {
    switch (n) {
        case 0: bulk_wait_read<0>(); break;
        case 1: bulk_wait_read<1>(); break;
        case 2: bulk_wait_read<2>(); break;
        case 3: bulk_wait_read<3>(); break;
        case 4: bulk_wait_read<4>(); break;
        case 5: bulk_wait_read<5>(); break;
        case 6: bulk_wait_read<6>(); break;
        default: bulk_wait_read<7>(); break;
    }
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


}  // namespace a2av
