// Combine: the return trip of the MoE exchange.  For every token the k expert
// outputs are gathered from the windows and summed with the gate weights:
//   out[s][t] = bf16_rne( sum_{j=0..k-1, slot>=0} w[s][t][j] * y[slot_map[s][t][j]] )
// accumulated in fp32 from +0 in slot order, each product and each sum
// rounded on its own, so the result does not depend on the launch shape.
// NCCLX pages: qiguanping deep dive section 7, Figure 13 (the dispatch
// shuffle and the combine).
//
// Work unit = one of `nsplit` pieces of one token's row (nsplit is chosen so
// that there are several units per warp: whole rows for many tokens, pieces
// for few), taken by the warps in a token-major grid stride, with 16-byte
// vector gathers of 32*U vectors per step.  The kernel is
// instantiated for k in {1, 2, 4, 8}, the slots taken in groups of G whose
// G*U loads are in flight together before their ordered accumulation; other
// k use the generic loop.
// Calls with fewer tokens than warps (decode-sized batches, rows split into
// pieces) run combine_batched_kernel, which loads the slot rows and gates of
// several units at once.  Launched as a programmatic dependent of the pack
// kernel.
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

// both values rounded to bf16 (nearest-even), lo into the low half-word: one
// cvt.rn.bf16x2.f32, which rounds each lane as cvt.rn.bf16.f32 does
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Eight fp32 accumulators.  The first slot that contributes goes through the
// packed two-lane fp32 FMA of the sm_100 family with a +0 addend: fma(w, y,
// +0) rounds only the product, and adding +0 is exact (it turns a -0 product
// into +0), so this is bit for bit the separately rounded product added to
// the +0 accumulator, one instruction per pair of values; slot 0 takes this
// path when it has a row.  Every other slot (slot 0 included, when it has no
// row and the accumulators stay +0) is a scalar __fmul_rn then __fadd_rn,
// which is correct whatever the accumulators hold: a packed multiply followed by a
// packed add is evaluated as one fused operation on this target (a device
// probe over 4M random triples matched fmaf in every case), which would drop
// the product's rounding.
__device__ __forceinline__ uint64_t pair_w(float w) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(w));
    return d;
}

// (lo, hi) = fma(w, (the two bf16 values of q, the low half-word first), +0)
__device__ __forceinline__ void first_pair(float &lo, float &hi, uint64_t w2, uint32_t q) {
    asm("{\n\t.reg .b32 l, h;\n\t.reg .b64 y, d;\n\t"
        "shl.b32 l, %2, 16;\n\tand.b32 h, %2, 0xffff0000;\n\tmov.b64 y, {l, h};\n\t"
        "fma.rn.f32x2 d, %3, y, %4;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(q), "l"(w2), "l"(0ull));
}

// one slot's eight values into the accumulators; `first`: the accumulators
// still hold +0 (then either path gives the same bits)
__device__ __forceinline__ void accumulate(float (&acc)[8], const uint4 &v, float w, bool first) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
    if (first) {
        const uint64_t w2 = pair_w(w);
#pragma unroll
        for (int i = 0; i < 4; ++i) first_pair(acc[2 * i], acc[2 * i + 1], w2, q[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16lo(q[i])));
            acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16hi(q[i])));
        }
    }
}

__device__ __forceinline__ uint4 to_bf16x8(const float (&acc)[8]) {
    return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                      pack_bf16x2(acc[6], acc[7]));
}

// One step of a unit: vectors [vb, min(vb + 32*U, vb_end)) of one token's
// row, gathered from its k slots, accumulated in slot order and stored to
// dst.  Lane m0 + j holds slot j's arena row (-1: no row) and gate weight.
// The k slots go in groups of G (G divides KT): the G*U loads of a group are
// in flight together, then accumulated in slot order before the next group's
// loads.  Fewer slots per group and more vectors per slot make each row
// access a longer contiguous run (U*512 bytes per warp), which the DRAM
// serves faster: for the r32 E256 T2048 H7168 top-8 combine, U=4 with one
// slot at a time (4 loads per lane, 80 registers) takes 1,285 us, U=4 G=2
// 1,286, U=2 G=2 1,290, U=2 G=4 1,360 and U=1 G=8 (all 8 slots at once)
// 1,324.
template <int KT, int U, int G = KT>
__device__ __forceinline__ void combine_step(int k, int lane, const char *y, size_t rowb, int32_t row, float w,
                                             int m0, int vb, int vb_end, char *dst) {
    float acc[U][8];
#pragma unroll
    for (int q = 0; q < U; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
    if constexpr (KT > 0) {
        static_assert(KT % G == 0, "slot groups divide k");
        int32_t rows[KT];
#pragma unroll
        for (int j = 0; j < KT; ++j) rows[j] = __shfl_sync(kFull, row, m0 + j);
#pragma unroll
        for (int g0 = 0; g0 < KT; g0 += G) {
            uint4 buf[G][U];
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const int v = vb + q * 32 + lane;
                    buf[jj][q] = make_uint4(0u, 0u, 0u, 0u);
                    if (rows[g0 + jj] >= 0 && v < vb_end)
                        buf[jj][q] = ld_stream_v4(y + (size_t)rows[g0 + jj] * rowb + (size_t)v * 16);
                }
            }
#pragma unroll
            for (int jj = 0; jj < G; ++jj) {
                const int j = g0 + jj;
                const float wj = __shfl_sync(kFull, w, m0 + j);
                if (rows[j] < 0) continue;  // warp-uniform: rows[] are the same in every lane
#pragma unroll
                for (int q = 0; q < U; ++q) accumulate(acc[q], buf[jj][q], wj, j == 0);
            }
        }
    } else {
        for (int j = 0; j < k; ++j) {
            const int32_t rj = __shfl_sync(kFull, row, m0 + j);
            const float wj = __shfl_sync(kFull, w, m0 + j);
            if (rj < 0) continue;
            uint4 buf[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int v = vb + q * 32 + lane;
                buf[q] = make_uint4(0u, 0u, 0u, 0u);
                if (v < vb_end) buf[q] = ld_stream_v4(y + (size_t)rj * rowb + (size_t)v * 16);
            }
#pragma unroll
            for (int q = 0; q < U; ++q) accumulate(acc[q], buf[q], wj, j == 0);
        }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
        const int v = vb + q * 32 + lane;
        if (v < vb_end) st_stream_v4(dst + (size_t)v * 16, to_bf16x8(acc[q]));
    }
}

template <int KT, int U, int G = (KT > 0 ? KT : 1)>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
    const Geometry &g = a.g;
    const int k = KT > 0 ? KT : g.k;
    const int lane = threadIdx.x & 31;
    const int nv = g.H >> 3;               // 16-byte vectors per row
    const int step = 32 * U;               // vectors per inner step
    const uint32_t nsplit = (uint32_t)a.nsplit;  // pieces per row (1 = whole-row units)
    const int steps_per_row = (nv + step - 1) / step;
    const int steps_per_unit = (steps_per_row + (int)nsplit - 1) / (int)nsplit;
    // 32-bit unit indices (a 64-bit divide is a subroutine call): units =
    // R*T*nsplit < 2^31, since R*T*k < 2^31 and nsplit > 1 only when R*T is
    // below four units per warp; unsigned, so that un + nw cannot overflow
    const uint32_t units = (uint32_t)g.R * (uint32_t)g.T * nsplit;
    const uint32_t T = (uint32_t)g.T;
    const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
    const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t rowb = (size_t)g.H * 2;
    const char *y = reinterpret_cast<const char *>(a.y);
    bool bad_slot = false;
    // Few-token calls: the next call's splits kernel (a programmatic
    // dependent) may take its SM slots now; its own dependency wait still
    // covers every store of this grid.
    if (a.trigger_early) grid_launch_dependents();
    grid_dependency_wait();  // slot_map and y come from the kernels before
    uint32_t cur = 0xffffffffu;
    int32_t row = -1;
    float w = 0.f;
    bool active = true;
    // token-major grid stride: the warps active at one time cover a compact
    // stretch of `out` (and of each token's gathered rows)
    for (uint32_t un = gw; un < units; un += nw) {
        const uint32_t u = un / nsplit;
        const int piece = (int)(un - u * nsplit);
        if (u != cur) {
            cur = u;
            const uint32_t s_tok = u / T;
            active = (int)(u - s_tok * T) < active_tokens(a.num_tokens, (int)s_tok, g.T);
            row = -1;
            w = 0.f;
            if (lane < k) {
                row = __ldg(a.slot_map + (size_t)u * k + lane);
                w = __ldg(a.gate + (size_t)u * k + lane);
                if (row >= a.arena_rows) {
                    bad_slot = true;
                    row = -1;
                }
            }
        }
        if (!active) continue;  // warp-uniform: the token takes no part, its out row is left alone
        char *dst = reinterpret_cast<char *>(a.out) + (size_t)u * rowb;
        const int vb_end = min(nv, (piece + 1) * steps_per_unit * step);
        for (int vb = piece * steps_per_unit * step; vb < vb_end; vb += step)
            combine_step<KT, U, G>(k, lane, y, rowb, row, w, 0, vb, vb_end, dst);
    }
    if (__any_sync(kFull, bad_slot) && lane == 0) atomicOr(a.status, kDevBadSlot);
}

// The same combine for calls with fewer tokens than warps, where every row is
// split into pieces and each warp has a few one-step units whose time is
// memory round trips: the slot rows and gate weights of the warp's next
// M = 32/k units come in with one warp-wide load (lane l: slot l % k of unit
// l / k) before any of their gathers, so each unit waits on one round trip
// instead of two (r8 E128 T256 H5120 top-1: 24.6 against 26.2 us per step).
// With whole-row units the plain kernel above is faster.
template <int KT, int U>
__global__ void __launch_bounds__(256) combine_batched_kernel(const CombineArgs a) {
    const Geometry &g = a.g;
    const int k = KT > 0 ? KT : g.k;
    const int lane = threadIdx.x & 31;
    const int nv = g.H >> 3;
    const int step = 32 * U;
    const uint32_t nsplit = (uint32_t)a.nsplit;
    const int steps_per_row = (nv + step - 1) / step;
    const int steps_per_unit = (steps_per_row + (int)nsplit - 1) / (int)nsplit;
    const uint32_t units = (uint32_t)g.R * (uint32_t)g.T * nsplit;  // < 2^31, as in combine_kernel
    const uint32_t T = (uint32_t)g.T;
    const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
    const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t rowb = (size_t)g.H * 2;
    const char *y = reinterpret_cast<const char *>(a.y);
    const int M = 32 / k;
    const int mi = lane / k, mj = lane - mi * k;
    bool bad_slot = false;
    if (a.trigger_early) grid_launch_dependents();  // as in combine_kernel
    grid_dependency_wait();
    // the warp's units are gw, gw + nw, ... (token-major, as in combine_kernel);
    // base + nw*M stays below 2^32 since units < 2^31 and nw*M <= 2048 per SM
    for (uint32_t base = gw; base < units; base += nw * (uint32_t)M) {
        int32_t mrow = -1;
        float mw = 0.f;
        int mact = 0;
        if (mi < M && base + (uint32_t)mi * nw < units) {
            const uint32_t u = (base + (uint32_t)mi * nw) / nsplit;
            const uint32_t s_tok = u / T;
            mact = (int)(u - s_tok * T) < active_tokens(a.num_tokens, (int)s_tok, g.T);
            mrow = __ldg(a.slot_map + (size_t)u * k + mj);
            mw = __ldg(a.gate + (size_t)u * k + mj);
            if (mrow >= a.arena_rows) {
                bad_slot = true;
                mrow = -1;
            }
        }
#pragma unroll 1
        for (int bi = 0; bi < M; ++bi) {
            const uint32_t un = base + (uint32_t)bi * nw;
            if (un >= units) break;                   // warp-uniform
            if (!__shfl_sync(kFull, mact, bi * k)) continue;  // warp-uniform: out row left alone
            const uint32_t u = un / nsplit;
            const int piece = (int)(un - u * nsplit);
            char *dst = reinterpret_cast<char *>(a.out) + (size_t)u * rowb;
            const int vb_end = min(nv, (piece + 1) * steps_per_unit * step);
            for (int vb = piece * steps_per_unit * step; vb < vb_end; vb += step)
                combine_step<KT, U>(k, lane, y, rowb, mrow, mw, bi * k, vb, vb_end, dst);
        }
    }
    if (__any_sync(kFull, bad_slot) && lane == 0) atomicOr(a.status, kDevBadSlot);
}

// ---------------------------------------------------------------------------
// TMA combine, warp-specialised (A2AV_FLAG_COMBINE_TMA).  Persistent grid,
// one CTA per SM by default, each owning a contiguous range of tokens split
// into work units (token, chunk of the row).  Warp 0 produces: for every
// unit its lane j issues one cp.async.bulk of slot j's row chunk into the
// unit's shared-memory stage (completion on the stage's `full` mbarrier) and
// records the slot mask and gate weights beside it.  Warps 1..NC consume:
// unit p goes to consumer p % NC, which accumulates the stage in slot order
// (fp32, each product and sum rounded on its own), streams the bf16 result
// to `out` and releases the stage on its `empty` mbarrier; the producer
// refills a stage only after that release.  The ring keeps up to
// `stages` * k * chunk bytes in flight per CTA, each load one contiguous
// chunk of a row, without holding registers for them.
//
// Every wait is bounded (a.wait_polls in the loops).  A warp whose wait
// gives up raises a CTA-wide abort flag and sets A2AV_DEV_WAIT_TIMEOUT; the
// others leave their loops at the flag; before the CTA exits, the producer
// waits (full bound) for the last unit it issued into every stage, so no
// bulk load is still writing this CTA's shared memory when it leaves.
// ---------------------------------------------------------------------------
struct StageMeta {
    uint32_t mask;  // bit j: slot j has a row in this stage
    uint32_t skip;  // 1: the unit's token takes no part (nothing loaded, nothing written)
    uint32_t pad[2];
    float w[kMaxTopk];
};

constexpr int kTmaConsumers = 8;  // consumer warps per CTA
constexpr int kTmaThreads = 32 * (1 + kTmaConsumers);

// Bounded wait on an mbarrier phase that also gives up as soon as another
// warp of the CTA has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, long long limit, volatile int *abort) {
    for (long long it = 0; it < limit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    return false;
}

__global__ void __launch_bounds__(kTmaThreads, 1) combine_tma_kernel(const CombineArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int abort_flag;
    const Geometry &g = a.g;
    const int k = g.k;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = a.stages, CH = a.chunk_bytes, nch = a.nchunks;
    const size_t stage_bytes = (size_t)k * CH;
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + (size_t)NS * stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + NS);
    uint64_t *empty = full + NS;
    volatile int *abort = &abort_flag;

    const long long ntok = (long long)g.R * g.T;
    const long long per = (ntok + gridDim.x - 1) / gridDim.x;
    const long long tb = min(ntok, (long long)blockIdx.x * per);
    const long long te = min(ntok, tb + per);
    if (tb >= te) return;  // the whole CTA
    const long long n = (te - tb) * nch;
    const size_t rowb = (size_t)g.H * 2;
    const char *y = reinterpret_cast<const char *>(a.y);
    char *outp = reinterpret_cast<char *>(a.out);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependency_wait();  // slot_map and y come from the kernels before

    long long issued = 0;  // producer: units issued so far
    bool bad_slot = false;
    if (warp == 0) {
        // slots and weights of a batch of BT tokens, one per lane
        const int BT = max(1, 32 / k);
        const int my_b = lane / k, my_j = lane - my_b * k;
        auto load_batch = [&](long long tok0, int32_t &row, float &w) {
            const long long tok = tok0 + my_b;
            row = -1;
            w = 0.f;
            if (my_b < BT && tok < te) {
                row = __ldg(a.slot_map + (size_t)tok * k + my_j);
                w = __ldg(a.gate + (size_t)tok * k + my_j);
            }
        };
        long long ib0 = tb;  // first token of the current batch
        int32_t cur_row, nxt_row;
        float cur_w, nxt_w;
        load_batch(ib0, cur_row, cur_w);
        load_batch(ib0 + BT, nxt_row, nxt_w);
        for (long long p = 0; p < n; ++p) {
            const int st = (int)(p % NS);
            if (p >= NS) {  // the consumer of unit p - NS has released the stage
                int ok = 1;
                if (lane == 0) ok = wait_or_abort(&empty[st], (uint32_t)((p / NS - 1) & 1), a.wait_polls, abort);
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) break;
            }
            const long long tok = tb + p / nch;
            if (tok >= ib0 + BT) {  // tokens only move forward
                ib0 += BT;
                cur_row = nxt_row;
                cur_w = nxt_w;
                load_batch(ib0 + BT, nxt_row, nxt_w);
            }
            const uint32_t off = (uint32_t)(p % nch) * CH;
            const uint32_t bytes = (uint32_t)min((size_t)CH, rowb - off);
            const int src = ((int)(tok - ib0) * k + (lane % k)) & 31;
            const int32_t r = __shfl_sync(kFull, cur_row, src);
            const float w = __shfl_sync(kFull, cur_w, src);
            const int s_tok = (int)(tok / g.T);
            const bool tok_active = tok - (long long)s_tok * g.T < active_tokens(a.num_tokens, s_tok, g.T);
            const bool in_arena = tok_active && r >= 0 && r < a.arena_rows;
            bad_slot |= lane < k && r >= a.arena_rows;
            const uint32_t mask = __ballot_sync(kFull, lane < k && in_arena);
            if (lane < k) meta[st].w[lane] = w;
            if (lane == 0) {
                meta[st].mask = mask;
                meta[st].skip = tok_active ? 0u : 1u;
            }
            // the consumer's generic reads of this stage precede the async refill
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(mask) * bytes);
            __syncwarp();
            if (lane < k && in_arena)
                bulk_load(smem + (size_t)st * stage_bytes + (size_t)lane * CH, y + (size_t)r * rowb + off, bytes,
                          &full[st]);
            issued = p + 1;
        }
        if (issued < n && lane == 0 && !*abort) {
            abort_flag = 1;
            atomicOr(a.status, kDevWaitTimeout);
        }
    } else {
        // Consumer c owns stages c, c + NCe, c + 2*NCe, ... (NS is a multiple
        // of NCe) and takes their units in order, so it never waits on a stage
        // more than one phase ahead of that stage's barrier: parity waits stay
        // unambiguous.  Consumers beyond the stage count have nothing to do.
        const int c = warp - 1;
        const int NCe = NS < kTmaConsumers ? NS : kTmaConsumers;
        for (long long p = c, base = 0; c < NCe && p < n;) {
            const int st = (int)(p % NS);
            int ok = 1;
            if (lane == 0) ok = wait_or_abort(&full[st], (uint32_t)((p / NS) & 1), a.wait_polls, abort);
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) {
                if (lane == 0 && atomicExch(&abort_flag, 1) == 0) atomicOr(a.status, kDevWaitTimeout);
                break;
            }
            const long long tok = tb + p / nch;
            const uint32_t off = (uint32_t)(p % nch) * CH;
            const int nvec = (int)(min((size_t)CH, rowb - off) >> 4);
            const uint32_t mask = meta[st].mask;
            const bool skip = meta[st].skip != 0u;
            const unsigned char *stage = smem + (size_t)st * stage_bytes;
            char *dst = outp + (size_t)tok * rowb + off;
            for (int v = lane; v < nvec && !skip; v += 32) {
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.f;
                for (int j = 0; j < k; ++j) {
                    if (!((mask >> j) & 1u)) continue;
                    const uint4 val = *reinterpret_cast<const uint4 *>(stage + (size_t)j * CH + (size_t)v * 16);
                    accumulate(acc, val, meta[st].w[j], j == 0);
                }
                st_stream_v4(dst + (size_t)v * 16, to_bf16x8(acc));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            // next unit of this consumer: its next stage in this round of NS
            // units, else its first stage in the next round
            p += NCe;
            if (p >= base + NS) {
                base += NS;
                p = base + c;
            }
        }
    }
    __syncthreads();
    // Leave only once every load issued into this CTA's shared memory has
    // landed: the last unit issued into each stage (earlier ones completed
    // before that stage could be refilled).  Full bound: in-bounds bulk copies
    // complete unless the context is already lost.
    if (warp == 0 && lane == 0)
        for (int st = 0; st < NS && st < issued; ++st) {
            const long long last = st + (long long)NS * ((issued - 1 - st) / NS);
            mbar_wait_bounded(&full[st], (uint32_t)((last / NS) & 1), kWaitLimit);
        }
    if (warp == 0 && __any_sync(kFull, bad_slot) && lane == 0) atomicOr(a.status, kDevBadSlot);
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

using CombineKernel = void (*)(const CombineArgs);

// The instantiated (k, U, G, batch) variants; U = 16-byte vectors per lane
// and slot, G = slots per load group, batch = combine_batched_kernel (top-1
// and top-2 only; G = k).
struct CombineVariant {
    int k, u, g;
    bool batch;
    CombineKernel fn;
};
const CombineVariant kCombineVariants[] = {
    {1, 2, 1, false, combine_kernel<1, 2>}, {1, 4, 1, false, combine_kernel<1, 4>},
    {1, 8, 1, false, combine_kernel<1, 8>},
    {2, 1, 2, false, combine_kernel<2, 1>}, {2, 2, 2, false, combine_kernel<2, 2>},
    {2, 4, 2, false, combine_kernel<2, 4>}, {2, 2, 1, false, combine_kernel<2, 2, 1>},
    {2, 4, 1, false, combine_kernel<2, 4, 1>},
    {4, 1, 4, false, combine_kernel<4, 1>}, {4, 2, 4, false, combine_kernel<4, 2>},
    {4, 2, 2, false, combine_kernel<4, 2, 2>}, {4, 4, 2, false, combine_kernel<4, 4, 2>},
    {4, 4, 1, false, combine_kernel<4, 4, 1>},
    {8, 1, 8, false, combine_kernel<8, 1>}, {8, 2, 4, false, combine_kernel<8, 2, 4>},
    {8, 2, 2, false, combine_kernel<8, 2, 2>}, {8, 4, 2, false, combine_kernel<8, 4, 2>},
    {8, 4, 1, false, combine_kernel<8, 4, 1>},
    {0, 1, 1, false, combine_kernel<0, 1>}, {0, 2, 1, false, combine_kernel<0, 2>},
    {1, 2, 1, true, combine_batched_kernel<1, 2>}, {1, 4, 1, true, combine_batched_kernel<1, 4>},
    {2, 2, 2, true, combine_batched_kernel<2, 2>},
};

// Measured on GB300: fewer loads per lane and more resident warps win
// (k*U of 2 to 8 vectors in flight per lane).  With the packed fp32
// arithmetic U=2 also wins for top-1 batches of few tokens (r8 T256 H5120:
// 25.6 vs 26.0 us per step with U=4), where the scalar code had preferred U=4.
// With batched metadata (fewer tokens than warps) U=4 wins for top-1 (r8 E128
// T256 H5120: 24.6 against 24.8 us per step with U=2, 26.2 us unbatched).
// Top-8: U=4, one slot at a time (see combine_step).  Top-2: U=2 with both
// slots at once equals U=2 one slot at a time (304.2 against 304.3 us on r16
// E128 T4096 H5120); U=4 loses (323 us one slot at a time, 380 us both).
int default_unroll(int k, bool batch) {
    switch (k) {
        case 1: return batch ? 4 : 2;
        case 2: return 2;
        case 4: return 1;
        case 8: return 4;
        default: return 1;
    }
}

// Slots per load group for a given unroll: about 4 loads in flight per
// lane (the measured defaults: top-8 U=4 G=1, top-2 U=2 G=2, top-4 U=1
// G=4).
int default_group(int k, int u) {
    int g = 4 / (u > 0 ? u : 1);
    if (g < 1) g = 1;
    return g < k ? g : k;
}

// Kernel for this plan's k and requested unroll / slot group (0: defaults;
// otherwise the nearest instantiated variant); nullptr if there is no
// batched kernel for k.
const CombineVariant *pick_variant(int k, int want_u, int want_g, bool batch) {
    const int kk = (k == 1 || k == 2 || k == 4 || k == 8) ? k : 0;
    const int u = want_u > 0 ? want_u : (kk ? default_unroll(kk, batch) : (batch ? 1 : 2));
    const int g = want_g > 0 ? want_g : (kk ? default_group(kk, u) : 1);
    const CombineVariant *best = nullptr;
    auto dist = [&](const CombineVariant &v) { return 16 * abs(v.u - u) + abs(v.g - g); };
    for (const auto &v : kCombineVariants) {
        if (v.k != kk || v.batch != batch) continue;
        if (!best || dist(v) < dist(*best) || (dist(v) == dist(*best) && v.u < best->u)) best = &v;
    }
    return best;
}

cudaError_t occupancy_grid(a2av_plan_s &p, const CombineVariant *v) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v->fn, 256, 0);
    p.combine.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    // split rows so that every warp gets at least ~4 units
    const long long warps = (long long)p.combine.grid * 8;
    const long long ntok = (long long)p.g.R * p.g.T;
    const int steps_per_row = ((p.g.H >> 3) + 32 * v->u - 1) / (32 * v->u);
    long long ns = (4 * warps + ntok - 1) / ntok;
    if (ns < 1) ns = 1;
    if (ns > steps_per_row) ns = steps_per_row;
    p.comb_nsplit = (int32_t)ns;
    p.comb_unroll = v->u;
    p.comb_group = v->g;
    p.comb_batch = v->batch;
    return e;
}

}  // namespace

constexpr int kCombStagesMax = 32;
// two CTAs per SM: 16 consumer warps (r32 top-8: 2,358 against 4,021 us with one)
constexpr int kCombDefaultCtasPerSm = 2;
constexpr int kCombDefaultStageBytes = 16384;

cudaError_t configure_combine_tma(a2av_plan_s &p) {
    const size_t rowb = (size_t)p.g.H * 2;
    const int cps = p.cfg.combine_ctas_per_sm > 0 ? p.cfg.combine_ctas_per_sm : kCombDefaultCtasPerSm;
    const size_t target = p.cfg.combine_stage_bytes > 0 ? (size_t)p.cfg.combine_stage_bytes : kCombDefaultStageBytes;
    size_t chunk = (target / (size_t)p.g.k) / 16 * 16;
    if (chunk < 256) chunk = 256;
    if (chunk > rowb) chunk = rowb;
    int max_optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.cfg.device);
    if (e != cudaSuccess) return e;
    size_t budget = (size_t)max_optin / cps;
    budget = budget > 2048 ? budget - 2048 : budget;
    // at least two stages: shrink the chunk if the requested one does not fit
    while (chunk > 256 && 2 * ((size_t)p.g.k * chunk + sizeof(StageMeta) + 16) > budget) chunk = (chunk / 2 + 15) / 16 * 16;
    const size_t per_stage = (size_t)p.g.k * chunk + sizeof(StageMeta) + 16;  // data, meta, full + empty barriers
    int stages = (int)(budget / per_stage);
    if (stages > kCombStagesMax) stages = kCombStagesMax;
    // every consumer warp owns the same number of stages (see the kernel)
    if (stages >= kTmaConsumers) stages = stages / kTmaConsumers * kTmaConsumers;
    if (stages < 2) return cudaErrorInvalidConfiguration;
    p.comb_chunk_bytes = (int32_t)chunk;
    p.comb_nchunks = (int32_t)((rowb + chunk - 1) / chunk);
    p.comb_stages = stages;
    p.combine.block = kTmaThreads;
    p.combine.grid = p.num_sms * cps;
    p.combine.smem = (size_t)stages * per_stage;
    // the cap on dynamic shared memory leaves room for the kernel's static
    // shared memory (its abort flag): static + dynamic may not exceed the opt-in
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, combine_tma_kernel);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(combine_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_optin - (int)fa.sharedSizeBytes);
}

cudaError_t configure_combine(a2av_plan_s &p) {
    p.combine.block = 256;
    p.scale.block = 256;
    cudaError_t e;
    if (p.cfg.flags & A2AV_FLAG_COMBINE_TMA) {
        p.combine_tma = 1;
        e = configure_combine_tma(p);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, expert_scale_kernel, 256, 0);
        p.scale.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
        return e;
    }
    p.combine_tma = 0;
    e = occupancy_grid(p, pick_variant(p.g.k, p.cfg.combine_unroll, 0, false));
    if (e != cudaSuccess) return e;
    // Fewer tokens than warps: the call is latency-bound.  The pack then lets
    // the combine's CTAs take their SM slots early, and where rows are split
    // into several pieces the combine batches its metadata loads.
    p.few_tokens = (long long)p.g.R * p.g.T < (long long)p.combine.grid * 8;
    const CombineVariant *vb = p.few_tokens ? pick_variant(p.g.k, p.cfg.combine_unroll, 0, true) : nullptr;
    if (vb && (p.g.H >> 3) > 32 * vb->u) {
        e = occupancy_grid(p, vb);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, expert_scale_kernel, 256, 0);
    p.scale.grid = p.num_sms * (per_sm > 0 ? per_sm : 1);
    return e;
}

cudaError_t launch_combine(const a2av_plan_s &p, const CombineArgs &a, cudaStream_t s) {
    cudaError_t e;
    CombineArgs b = a;
    if (p.combine_tma) {
        b.chunk_bytes = p.comb_chunk_bytes;
        b.nchunks = p.comb_nchunks;
        b.stages = p.comb_stages;
        b.wait_polls = p.wait_polls;
        e = launch_pdl(combine_tma_kernel, p.combine.grid, p.combine.block, p.combine.smem, s, b);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    b.nsplit = p.comb_nsplit;
    b.trigger_early = p.few_tokens ? 1 : 0;
    e = launch_pdl(pick_variant(p.g.k, p.comb_unroll, p.comb_group, p.comb_batch)->fn, p.combine.grid, 256, 0, s, b);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_scale(const a2av_plan_s &p, const ScaleArgs &a, cudaStream_t s) {
    expert_scale_kernel<<<p.scale.grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace a2av
