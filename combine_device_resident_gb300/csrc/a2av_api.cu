// C ABI of the device-resident dispatch/combine data plane: validation, plans,
// and the enqueueing calls.  All allocation happens in a2av_plan_create; the
// enqueueing calls only launch kernels on the caller's stream (no sync, no
// allocation, no device-to-host reads), so they can be captured in a CUDA
// graph and replayed while the routing in device memory changes.
#include <stdio.h>
#include <string.h>

#include <new>

#include "a2av_internal.cuh"

namespace {

thread_local char g_last_error[256] = "";

a2av_status_t cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
    return A2AV_ERR_CUDA;
}

// Makes the plan's device current for the duration of a call and restores the
// caller's device afterwards.
struct DeviceGuard {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
        else if (err == cudaSuccess) prev = -1;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

bool aligned(const void *p, size_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// recv_expert_offsets: required in the expert-grouped order, optional otherwise.
bool splits_ok(const a2av_plan_s *p, const a2av_splits_t *sp) {
    if (!sp) return false;
    const bool reo_ok = sp->recv_expert_offsets ? aligned(sp->recv_expert_offsets, 4)
                                                : p->cfg.recv_order != A2AV_ORDER_EXPERT;
    return reo_ok && aligned(sp->send_counts, 4) && aligned(sp->send_offsets, 4) && aligned(sp->recv_counts, 4) &&
           aligned(sp->recv_offsets, 4) && aligned(sp->recv_expert_counts, 4) && aligned(sp->recv_total, 4) &&
           aligned(sp->window_base, 4);
}

a2av::Splits to_internal(const a2av_splits_t *sp) {
    return a2av::Splits{sp->send_counts,        sp->send_offsets, sp->recv_counts,  sp->recv_offsets,
                        sp->recv_expert_counts, sp->recv_total,   sp->window_base, sp->recv_expert_offsets};
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t row_bytes(const a2av_plan_s *p) { return (size_t)p->g.H * 2; }
size_t tokens(const a2av_plan_s *p) { return (size_t)p->g.R * p->g.T; }

}  // namespace

namespace a2av {
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
}  // namespace a2av

extern "C" {

a2av_status_t a2av_config_check(const a2av_config_t *c) {
    if (!c) return A2AV_ERR_INVALID_ARG;
    if (c->num_ranks < 1 || c->num_ranks > a2av::kMaxRanks) return A2AV_ERR_INVALID_ARG;
    if (c->num_experts < c->num_ranks || c->num_experts > a2av::kMaxExperts) return A2AV_ERR_INVALID_ARG;
    if (c->num_experts % c->num_ranks != 0) return A2AV_ERR_INVALID_ARG;
    if (c->tokens_per_rank < 1) return A2AV_ERR_INVALID_ARG;
    if (c->hidden < 8 || c->hidden % 8 != 0) return A2AV_ERR_INVALID_ARG;
    if (c->topk < 1 || c->topk > a2av::kMaxTopk) return A2AV_ERR_INVALID_ARG;
    const long long assignments = (long long)c->num_ranks * c->tokens_per_rank * c->topk;
    if (assignments >= (1ll << 31)) return A2AV_ERR_INVALID_ARG;
    if ((long long)c->tokens_per_rank * c->topk >= (1ll << 31) - a2av::kHistTile) return A2AV_ERR_INVALID_ARG;
    if (c->window_mode == A2AV_WINDOW_FIXED) {
        if (c->window_rows < 0 || (long long)c->num_ranks * c->window_rows >= (1ll << 31)) return A2AV_ERR_INVALID_ARG;
    } else if (c->window_mode == A2AV_WINDOW_PADDED) {
        if (assignments * c->num_ranks >= (1ll << 31)) return A2AV_ERR_INVALID_ARG;
    } else if (c->window_mode != A2AV_WINDOW_PACKED) {
        return A2AV_ERR_INVALID_ARG;
    }
    if (c->device < 0) return A2AV_ERR_INVALID_ARG;
    if (c->flags & ~(uint32_t)(A2AV_FLAG_PACK_LSU | A2AV_FLAG_SPLITS_TILED | A2AV_FLAG_COMBINE_TMA |
                               A2AV_FLAG_ROUTE_FUSED | A2AV_FLAG_ROUTE_WARP))
        return A2AV_ERR_INVALID_ARG;
    if (c->pack_store_lag < 0 || c->pack_store_lag > 8) return A2AV_ERR_INVALID_ARG;
    if (c->combine_ctas_per_sm < 0 || c->combine_ctas_per_sm > 8) return A2AV_ERR_INVALID_ARG;
    if (c->combine_stage_bytes < 0 || c->combine_stage_bytes % 16 != 0 || c->combine_stage_bytes > 131072)
        return A2AV_ERR_INVALID_ARG;
    if (c->combine_unroll < 0 || c->combine_unroll > 8) return A2AV_ERR_INVALID_ARG;
    if (c->pack_ctas_per_sm < 0 || c->pack_ctas_per_sm > 4) return A2AV_ERR_INVALID_ARG;
    if (c->pack_stage_bytes < 0 || c->pack_stage_bytes % 16 != 0 || c->pack_stage_bytes > 65536)
        return A2AV_ERR_INVALID_ARG;
    if (c->recv_order != A2AV_ORDER_SOURCE && c->recv_order != A2AV_ORDER_EXPERT) return A2AV_ERR_INVALID_ARG;
    if (c->recv_order == A2AV_ORDER_EXPERT && c->window_mode == A2AV_WINDOW_PADDED) return A2AV_ERR_INVALID_ARG;
    return A2AV_OK;
}

int64_t a2av_recv_arena_rows(const a2av_config_t *c) {
    if (a2av_config_check(c) != A2AV_OK) return -1;
    if (c->window_mode == A2AV_WINDOW_FIXED) return (int64_t)c->num_ranks * c->window_rows;
    if (c->window_mode == A2AV_WINDOW_PADDED)
        return (int64_t)c->num_ranks * c->num_ranks * c->tokens_per_rank * c->topk;
    return (int64_t)c->num_ranks * c->tokens_per_rank * c->topk;
}

a2av_status_t a2av_plan_create(const a2av_config_t *cfg, a2av_plan_t *out_plan) {
    if (!out_plan) return A2AV_ERR_INVALID_ARG;
    *out_plan = nullptr;
    a2av_status_t st = a2av_config_check(cfg);
    if (st != A2AV_OK) {
        snprintf(g_last_error, sizeof g_last_error, "invalid configuration");
        return st;
    }
    DeviceGuard guard(cfg->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");

    a2av_plan_s *p = new (std::nothrow) a2av_plan_s();
    if (!p) return A2AV_ERR_NO_MEMORY;
    p->cfg = *cfg;
    a2av::Geometry &g = p->g;
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
    p->pack_tma = (cfg->flags & A2AV_FLAG_PACK_LSU) ? 0 : 1;

    cudaError_t e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "cudaDeviceGetAttribute");
    }

    // Workspace: tile bases [R][tiles][E], per-rank totals [R], counters [R+1], status.
    const size_t n_tile = (size_t)g.R * g.tiles * g.E;
    const size_t off_tot = ((n_tile * 4) + 255) / 256 * 256;
    const size_t off_cnt = off_tot + (((size_t)g.R * 4) + 255) / 256 * 256;
    const size_t off_status = off_cnt + (((size_t)g.R + 1) * 4 + 255) / 256 * 256;
    p->workspace_bytes = off_status + 256;
    e = cudaMalloc(&p->workspace, p->workspace_bytes);
    if (e != cudaSuccess) {
        delete p;
        cuda_fail(e, "cudaMalloc(workspace)");
        return A2AV_ERR_NO_MEMORY;
    }
    char *base = static_cast<char *>(p->workspace);
    p->tile_base = reinterpret_cast<int32_t *>(base);
    p->rank_total = reinterpret_cast<int32_t *>(base + off_tot);
    p->counters = reinterpret_cast<uint32_t *>(base + off_cnt);
    p->status = reinterpret_cast<uint32_t *>(base + off_status);
    e = cudaMemset(p->workspace, 0, p->workspace_bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = a2av::configure_hist(*p);
    if (e == cudaSuccess) e = a2av::configure_pack(*p);
    if (e == cudaSuccess) e = a2av::configure_combine(*p);
    if (e == cudaSuccess) e = a2av::configure_route(*p);
    p->last_rows_final = p->splits_small;
    if (e != cudaSuccess) {
        cudaFree(p->workspace);
        delete p;
        return cuda_fail(e, "plan configuration");
    }
    *out_plan = p;
    return A2AV_OK;
}

a2av_status_t a2av_plan_destroy(a2av_plan_t p) {
    if (!p) return A2AV_OK;
    DeviceGuard guard(p->cfg.device);
    cudaError_t e = cudaFree(p->workspace);
    delete p;
    return e == cudaSuccess ? A2AV_OK : cuda_fail(e, "cudaFree(workspace)");
}

a2av_status_t a2av_splits(a2av_plan_t p, const int32_t *topk_idx, const a2av_splits_t *splits, int32_t *slot_map,
                          void *stream) {
    if (!p || !aligned(topk_idx, 4) || !aligned(slot_map, 4) || !splits_ok(p, splits)) return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::HistArgs a;
    memset(&a, 0, sizeof a);
    a.g = p->g;
    a.num_tokens = p->num_tokens;
    a.idx = topk_idx;
    a.slot_map = slot_map;
    a.tile_base = p->tile_base;
    a.rank_total = p->rank_total;
    a.counters = p->counters;
    a.status = p->status;
    a.sp = to_internal(splits);
    cudaError_t e = a2av::launch_hist(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "splits kernel launch");
    p->launches += 1;
    p->last_rows_final = p->splits_small;
    return A2AV_OK;
}

static a2av_status_t pack_into(a2av_plan_t p, const void *x, const int32_t *topk_idx, const a2av_splits_t *splits,
                               void *dst, int32_t *slot_map, void *stream, bool padded);

a2av_status_t a2av_pack(a2av_plan_t p, const void *x, const int32_t *topk_idx, const a2av_splits_t *splits,
                        void *recv, int32_t *slot_map, void *stream) {
    if (!p || p->cfg.window_mode == A2AV_WINDOW_PADDED) {
        a2av::set_last_error("a2av_pack: padded plans use a2av_pack_padded");
        return A2AV_ERR_INVALID_ARG;
    }
    return pack_into(p, x, topk_idx, splits, recv, slot_map, stream, false);
}

a2av_status_t a2av_pack_padded(a2av_plan_t p, const void *x, const int32_t *topk_idx, const a2av_splits_t *splits,
                               void *sendbuf, int32_t *slot_map, void *stream) {
    if (!p || p->cfg.window_mode != A2AV_WINDOW_PADDED) {
        a2av::set_last_error("a2av_pack_padded: the plan is not padded");
        return A2AV_ERR_INVALID_ARG;
    }
    return pack_into(p, x, topk_idx, splits, sendbuf, slot_map, stream, true);
}

static a2av_status_t pack_into(a2av_plan_t p, const void *x, const int32_t *topk_idx, const a2av_splits_t *splits,
                               void *recv, int32_t *slot_map, void *stream, bool padded) {
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(topk_idx, 4) || !aligned(slot_map, 4) ||
        !splits_ok(p, splits))
        return A2AV_ERR_INVALID_ARG;
    const int64_t rows = a2av_recv_arena_rows(&p->cfg);
    if (overlap(x, tokens(p) * row_bytes(p), recv, (size_t)rows * row_bytes(p))) return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::PackArgs a;
    memset(&a, 0, sizeof a);
    a.g = p->g;
    a.num_tokens = p->num_tokens;
    a.x = static_cast<const uint16_t *>(x);
    a.idx = topk_idx;
    a.slot_map = slot_map;
    a.tile_base = p->tile_base;
    a.send_offsets = splits->send_offsets;
    a.recv_offsets = splits->recv_offsets;
    a.window_base = splits->window_base;
    a.recv_expert_offsets = splits->recv_expert_offsets;
    a.recv = static_cast<uint16_t *>(recv);
    a.status = p->status;
    a.padded_tk = padded ? (int64_t)p->g.T * p->g.k : 0;
    a.rows_final = p->last_rows_final;
    cudaError_t e = a2av::launch_pack(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pack kernel launch");
    p->launches += 1;
    return A2AV_OK;
}

a2av_status_t a2av_exchange_padded(a2av_plan_t p, const void *sendbuf, void *recv, void *stream) {
    if (!p || p->cfg.window_mode != A2AV_WINDOW_PADDED || !aligned(sendbuf, 16) || !aligned(recv, 16))
        return A2AV_ERR_INVALID_ARG;
    const size_t bytes = (size_t)a2av_recv_arena_rows(&p->cfg) * row_bytes(p);
    if (overlap(sendbuf, bytes, recv, bytes)) return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::ExchangeArgs a;
    a.sendbuf = static_cast<const uint16_t *>(sendbuf);
    a.recv = static_cast<uint16_t *>(recv);
    a.R = p->g.R;
    a.block_vecs = (int64_t)p->g.T * p->g.k * (p->g.H / 8);
    cudaError_t e = a2av::launch_exchange_padded(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "padded exchange kernel launch");
    p->launches += 1;
    return A2AV_OK;
}

a2av_status_t a2av_dispatch_padded(a2av_plan_t p, const void *x, const int32_t *topk_idx,
                                   const a2av_splits_t *splits, void *sendbuf, void *recv, int32_t *slot_map,
                                   void *stream) {
    if (!p || p->cfg.window_mode != A2AV_WINDOW_PADDED || !aligned(sendbuf, 16) || !aligned(recv, 16))
        return A2AV_ERR_INVALID_ARG;
    const size_t bytes = (size_t)a2av_recv_arena_rows(&p->cfg) * row_bytes(p);
    if (overlap(x, tokens(p) * row_bytes(p), recv, bytes) || overlap(sendbuf, bytes, recv, bytes))
        return A2AV_ERR_INVALID_ARG;
    a2av_status_t st = a2av_splits(p, topk_idx, splits, slot_map, stream);
    if (st == A2AV_OK) st = a2av_pack_padded(p, x, topk_idx, splits, sendbuf, slot_map, stream);
    if (st == A2AV_OK) st = a2av_exchange_padded(p, sendbuf, recv, stream);
    return st;
}

a2av_status_t a2av_dispatch(a2av_plan_t p, const void *x, const int32_t *topk_idx, const a2av_splits_t *splits,
                            void *recv, int32_t *slot_map, void *stream) {
    if (p && p->cfg.window_mode == A2AV_WINDOW_PADDED) {
        a2av::set_last_error("a2av_dispatch: padded plans use a2av_dispatch_padded");
        return A2AV_ERR_INVALID_ARG;
    }
    if (!p || !aligned(x, 16) || !aligned(recv, 16) || !aligned(topk_idx, 4) || !aligned(slot_map, 4) ||
        !splits_ok(p, splits))
        return A2AV_ERR_INVALID_ARG;
    const int64_t rows = a2av_recv_arena_rows(&p->cfg);
    if (overlap(x, tokens(p) * row_bytes(p), recv, (size_t)rows * row_bytes(p))) return A2AV_ERR_INVALID_ARG;
    a2av_status_t st = a2av_splits(p, topk_idx, splits, slot_map, stream);
    if (st != A2AV_OK) return st;
    return a2av_pack(p, x, topk_idx, splits, recv, slot_map, stream);
}

a2av_status_t a2av_combine(a2av_plan_t p, const void *y, const float *gate_w, const int32_t *slot_map, void *out,
                           void *stream) {
    if (!p || !aligned(y, 16) || !aligned(out, 16) || !aligned(gate_w, 4) || !aligned(slot_map, 4))
        return A2AV_ERR_INVALID_ARG;
    const int64_t rows = a2av_recv_arena_rows(&p->cfg);
    if (overlap(y, (size_t)rows * row_bytes(p), out, tokens(p) * row_bytes(p))) return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::CombineArgs a;
    a.g = p->g;
    a.num_tokens = p->num_tokens;
    a.y = static_cast<const uint16_t *>(y);
    a.gate = gate_w;
    a.slot_map = slot_map;
    a.out = static_cast<uint16_t *>(out);
    a.arena_rows = rows;
    a.status = p->status;
    cudaError_t e = a2av::launch_combine(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    p->launches += 1;
    return A2AV_OK;
}

a2av_status_t a2av_expert_scale(a2av_plan_t p, const void *recv, const int32_t *topk_idx, const int32_t *slot_map,
                                void *y, void *stream) {
    if (!p || !aligned(recv, 16) || !aligned(y, 16) || !aligned(topk_idx, 4) || !aligned(slot_map, 4))
        return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::ScaleArgs a;
    a.g = p->g;
    a.recv = static_cast<const uint16_t *>(recv);
    a.idx = topk_idx;
    a.slot_map = slot_map;
    a.y = static_cast<uint16_t *>(y);
    a.arena_rows = a2av_recv_arena_rows(&p->cfg);
    a.status = p->status;
    cudaError_t e = a2av::launch_scale(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "expert scale kernel launch");
    p->launches += 1;
    return A2AV_OK;
}

a2av_status_t a2av_read_device_status(a2av_plan_t p, uint32_t *bits, int clear, void *stream) {
    if (!p || !bits) return A2AV_ERR_INVALID_ARG;
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(bits, p->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear) {
        e = cudaMemsetAsync(p->status, 0, sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e == cudaSuccess ? A2AV_OK : cuda_fail(e, "read device status");
}

a2av_status_t a2av_route(a2av_plan_t p, const float *logits, int32_t *topk_idx, float *gate_w, void *stream) {
    if (!p || !aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(gate_w, 4)) return A2AV_ERR_INVALID_ARG;
    if (p->g.k > p->g.E) {
        a2av::set_last_error("a2av_route: k distinct experts need k <= E");
        return A2AV_ERR_INVALID_ARG;
    }
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::RouteArgs a;
    a.g = p->g;
    a.num_tokens = p->num_tokens;
    a.logits = logits;
    a.idx = topk_idx;
    a.gate = gate_w;
    a.status = p->status;
    a.wait_polls = p->wait_polls;
    a.rsw = 0;  // set by launch_route for the lane-per-token kernel
    cudaError_t e = a2av::launch_route(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "route kernel launch");
    p->launches += 1;
    return A2AV_OK;
}

a2av_status_t a2av_route_splits(a2av_plan_t p, const float *logits, int32_t *topk_idx, float *gate_w,
                                const a2av_splits_t *splits, int32_t *slot_map, void *stream) {
    if (!p || !aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(gate_w, 4) || !aligned(slot_map, 4) ||
        !splits_ok(p, splits))
        return A2AV_ERR_INVALID_ARG;
    if (p->g.k > p->g.E) {
        a2av::set_last_error("a2av_route_splits: k distinct experts need k <= E");
        return A2AV_ERR_INVALID_ARG;
    }
    if (!(p->cfg.flags & A2AV_FLAG_ROUTE_FUSED) || !a2av::routed_splits_supported(*p)) {  // the two kernels
        a2av_status_t st = a2av_route(p, logits, topk_idx, gate_w, stream);
        return st == A2AV_OK ? a2av_splits(p, topk_idx, splits, slot_map, stream) : st;
    }
    DeviceGuard guard(p->cfg.device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    a2av::HistArgs a;
    memset(&a, 0, sizeof a);
    a.g = p->g;
    a.num_tokens = p->num_tokens;
    a.idx = topk_idx;
    a.slot_map = slot_map;
    a.tile_base = p->tile_base;
    a.rank_total = p->rank_total;
    a.counters = p->counters;
    a.status = p->status;
    a.sp = to_internal(splits);
    a.logits = logits;
    a.idx_out = topk_idx;
    a.gate_out = gate_w;
    cudaError_t e = a2av::launch_routed_hist(*p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "routed splits kernel launch");
    p->launches += 1;
    p->last_rows_final = 0;
    return A2AV_OK;
}

a2av_status_t a2av_set_active_tokens(a2av_plan_t p, const int32_t *num_tokens) {
    if (!p || (num_tokens && (reinterpret_cast<uintptr_t>(num_tokens) % 4) != 0)) return A2AV_ERR_INVALID_ARG;
    p->num_tokens = num_tokens;
    return A2AV_OK;
}

a2av_status_t a2av_set_wait_limit(a2av_plan_t p, int64_t polls) {
    if (!p) return A2AV_ERR_INVALID_ARG;
    p->wait_polls = polls < 0 ? a2av::kWaitLimit : (polls > a2av::kWaitLimit ? a2av::kWaitLimit : polls);
    return A2AV_OK;
}

const void *a2av_device_status_ptr(a2av_plan_t p) { return p ? p->status : nullptr; }

int64_t a2av_plan_launches(a2av_plan_t p) { return p ? p->launches : -1; }

const char *a2av_status_string(a2av_status_t s) {
    switch (s) {
        case A2AV_OK: return "ok";
        case A2AV_ERR_INVALID_ARG: return "invalid argument";
        case A2AV_ERR_CUDA: return "CUDA error";
        case A2AV_ERR_NO_MEMORY: return "out of device memory";
    }
    return "unknown status";
}

const char *a2av_last_error(void) { return g_last_error; }

}  // extern "C"
