// Dispatch without any allocation: a2av_dispatch_static.
//
// Some callers cannot call cudaMalloc where they dispatch: code inside a
// framework whose caching allocator owns all device memory and must not be
// bypassed, processes that run under a fixed device-memory budget that is
// spent by the time this library runs, and latency-critical loops that must
// not take cudaMalloc's implicit device synchronisation.  For them this entry
// point keeps its scratch (the per-tile histogram bases, the per-rank totals
// and the completion counters the splits kernel needs) in one file-scope
// __device__ array, so the only device memory it touches besides the
// caller's buffers is memory the library already owns from the moment it is
// loaded.
//
// The same splits and pack kernels as a2av_dispatch run; only where their
// scratch lives differs.  The array is shared by every call in the process,
// and every GPU that loads the library holds a copy of it until the process
// exits.  Per device, the first call does the set-up (the array's device
// address, the kernels' shared-memory attributes); per configuration, the
// first call computes the launch shapes; both are kept for later calls.
#include <stdio.h>

#include <mutex>

#include "a2av_internal.cuh"

namespace {

// 1 MiB of scratch per GPU (262144 int32).  Enough for, e.g., R=32 ranks,
// E=256 experts and 16384 assignments per rank (about 66k entries).
constexpr size_t kStaticScratchInts = 262144;
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int32_t *g_scratch_addr[kMaxDevices];  // device address of the array, per device
int g_num_sms[kMaxDevices];

size_t round64(size_t n) { return (n + 63) / 64 * 64; }

// Launch shapes of one configuration on one device, computed by the first
// call that uses them (configure_hist / configure_pack: kernel attributes,
// occupancy and cluster-residency queries) and reused by later calls.
struct ShapeEntry {
    bool used = false;
    a2av_config_t cfg{};
    a2av::LaunchShape hist, pack;
    int splits_small = 0;
    int32_t pack_chunk_bytes = 0, pack_nchunks = 0, pack_stages = 0, pack_lag = 1;
    int pack_stream_rows = 0;
};
constexpr int kShapeCache = 32;
ShapeEntry g_shapes[kShapeCache];
int g_next_shape = 0;  // round-robin replacement once the cache is full

bool same_config(const a2av_config_t &a, const a2av_config_t &b) {
    return a.num_ranks == b.num_ranks && a.num_experts == b.num_experts && a.tokens_per_rank == b.tokens_per_rank &&
           a.hidden == b.hidden && a.topk == b.topk && a.window_mode == b.window_mode &&
           a.window_rows == b.window_rows && a.device == b.device && a.flags == b.flags &&
           a.pack_ctas_per_sm == b.pack_ctas_per_sm && a.pack_stage_bytes == b.pack_stage_bytes &&
           a.pack_store_lag == b.pack_store_lag && a.combine_ctas_per_sm == b.combine_ctas_per_sm &&
           a.combine_stage_bytes == b.combine_stage_bytes && a.combine_unroll == b.combine_unroll &&
           a.recv_order == b.recv_order;
}

// One-time set-up of `dev` (with `dev` current): the array's device address
// and the SM count.  A later cudaDeviceReset is not supported: the address
// would belong to the destroyed context.
cudaError_t device_setup_locked(int dev) {
    if (g_scratch_addr[dev]) return cudaSuccess;
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_dispatch_scratch);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t *>(ptr);
    return cudaSuccess;
}

// Fills p's device fields (scratch address, SM count) and launch shapes for
// p.cfg, doing the device set-up and the shape configuration only the first
// time they are needed.
cudaError_t prepare(a2av_plan_s &p, int32_t **scratch) {
    const int dev = p.cfg.device;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    cudaError_t e = device_setup_locked(dev);
    if (e != cudaSuccess) return e;
    *scratch = g_scratch_addr[dev];
    p.num_sms = g_num_sms[dev];
    for (const ShapeEntry &s : g_shapes) {
        if (s.used && same_config(s.cfg, p.cfg)) {
            p.hist = s.hist;
            p.pack = s.pack;
            p.splits_small = s.splits_small;
            p.pack_chunk_bytes = s.pack_chunk_bytes;
            p.pack_nchunks = s.pack_nchunks;
            p.pack_stages = s.pack_stages;
            p.pack_lag = s.pack_lag;
            p.pack_stream_rows = s.pack_stream_rows;
            return cudaSuccess;
        }
    }
    e = a2av::configure_hist(p);
    if (e == cudaSuccess) e = a2av::configure_pack(p);
    if (e != cudaSuccess) return e;
    ShapeEntry &s = g_shapes[g_next_shape];
    g_next_shape = (g_next_shape + 1) % kShapeCache;
    s.used = true;
    s.cfg = p.cfg;
    s.hist = p.hist;
    s.pack = p.pack;
    s.splits_small = p.splits_small;
    s.pack_chunk_bytes = p.pack_chunk_bytes;
    s.pack_nchunks = p.pack_nchunks;
    s.pack_stages = p.pack_stages;
    s.pack_lag = p.pack_lag;
    s.pack_stream_rows = p.pack_stream_rows;
    return cudaSuccess;
}

bool aligned(const void *p, size_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" a2av_status_t a2av_dispatch_static(const a2av_config_t *cfg, const void *x, const int32_t *topk_idx,
                                              const a2av_splits_t *splits, void *recv, int32_t *slot_map,
                                              uint32_t *dev_status, void *stream) {
    if (a2av_config_check(cfg) != A2AV_OK || cfg->window_mode == A2AV_WINDOW_PADDED) {
        a2av::set_last_error("a2av_dispatch_static: invalid configuration (padded plans need a send buffer)");
        return A2AV_ERR_INVALID_ARG;
    }
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(topk_idx, 4) || !aligned(slot_map, 4) ||
        !aligned(dev_status, 4) || !splits || !aligned(splits->send_counts, 4) || !aligned(splits->send_offsets, 4) ||
        !aligned(splits->recv_counts, 4) || !aligned(splits->recv_offsets, 4) ||
        !aligned(splits->recv_expert_counts, 4) || !aligned(splits->recv_total, 4) ||
        !aligned(splits->window_base, 4) ||
        (splits->recv_expert_offsets ? !aligned(splits->recv_expert_offsets, 4)
                                     : cfg->recv_order == A2AV_ORDER_EXPERT)) {
        a2av::set_last_error("a2av_dispatch_static: null or misaligned pointer");
        return A2AV_ERR_INVALID_ARG;
    }

    a2av_plan_s p;  // host-side description only; nothing is allocated
    p.cfg = *cfg;
    a2av::Geometry &g = p.g;
    g.R = cfg->num_ranks;
    g.E = cfg->num_experts;
    g.T = cfg->tokens_per_rank;
    g.H = cfg->hidden;
    g.k = cfg->topk;
    g.epr = g.E / g.R;
    g.key_bits = 1;
    while ((1 << g.key_bits) <= g.E) ++g.key_bits;
    g.tiles = (int32_t)(((long long)g.T * g.k + a2av::kHistTile - 1) / a2av::kHistTile);
    g.window_mode = cfg->window_mode;
    g.recv_order = cfg->recv_order;
    g.window_rows = cfg->window_mode == A2AV_WINDOW_FIXED ? cfg->window_rows : 0;
    p.pack_tma = (cfg->flags & A2AV_FLAG_PACK_LSU) ? 0 : 1;

    const size_t row_bytes = (size_t)g.H * 2;
    const size_t x_bytes = (size_t)g.R * g.T * row_bytes;
    const size_t recv_bytes = (size_t)a2av_recv_arena_rows(cfg) * row_bytes;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ra = reinterpret_cast<uintptr_t>(recv);
    if (xa < ra + recv_bytes && ra < xa + x_bytes) {
        a2av::set_last_error("a2av_dispatch_static: recv overlaps x");
        return A2AV_ERR_INVALID_ARG;
    }

    const size_t n_tile = round64((size_t)g.R * g.tiles * g.E);
    const size_t n_tot = round64((size_t)g.R);
    const size_t n_cnt = round64((size_t)g.R + 1);
    if (n_tile + n_tot + n_cnt > kStaticScratchInts) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "a2av_dispatch_static: this shape needs %zu int32 of scratch, the static array holds %zu "
                 "(use a plan and a2av_dispatch instead)",
                 n_tile + n_tot + n_cnt, kStaticScratchInts);
        a2av::set_last_error(msg);
        return A2AV_ERR_INVALID_ARG;
    }

    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e == cudaSuccess && prev != cfg->device) e = cudaSetDevice(cfg->device);
    int32_t *scratch = nullptr;
    if (e == cudaSuccess) e = prepare(p, &scratch);
    if (e == cudaSuccess) {
        p.tile_base = scratch;
        p.rank_total = scratch + n_tile;
        p.counters = reinterpret_cast<uint32_t *>(scratch + n_tile + n_tot);
        p.status = dev_status;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The completion counters must start at zero; the previous call leaves them
    // at zero, but clear them anyway so that nothing depends on earlier calls.
    if (e == cudaSuccess) e = cudaMemsetAsync(p.counters, 0, ((size_t)g.R + 1) * sizeof(uint32_t), s);
    if (e == cudaSuccess) {
        a2av::HistArgs h{};
        h.g = g;
        h.num_tokens = nullptr;
        h.idx = topk_idx;
        h.slot_map = slot_map;
        h.tile_base = p.tile_base;
        h.rank_total = p.rank_total;
        h.counters = p.counters;
        h.status = dev_status;
        h.sp = a2av::Splits{splits->send_counts, splits->send_offsets, splits->recv_counts, splits->recv_offsets,
                            splits->recv_expert_counts, splits->recv_total, splits->window_base,
                            splits->recv_expert_offsets};
        e = a2av::launch_hist(p, h, s);
    }
    if (e == cudaSuccess) {
        a2av::PackArgs a{};
        a.g = g;
        a.x = static_cast<const uint16_t *>(x);
        a.idx = topk_idx;
        a.slot_map = slot_map;
        a.tile_base = p.tile_base;
        a.send_offsets = splits->send_offsets;
        a.recv_offsets = splits->recv_offsets;
        a.window_base = splits->window_base;
        a.recv_expert_offsets = splits->recv_expert_offsets;
        a.recv = static_cast<uint16_t *>(recv);
        a.status = dev_status;
        a.rows_final = p.splits_small;
        e = a2av::launch_pack(p, a, s);
    }
    if (prev >= 0 && prev != cfg->device) cudaSetDevice(prev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "a2av_dispatch_static: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
        a2av::set_last_error(msg);
        return A2AV_ERR_CUDA;
    }
    return A2AV_OK;
}
