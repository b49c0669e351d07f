// moe_a2a.cpp -- the C ABI declared in include/moe_a2a.h: configuration
// checks, workspace layout, the dispatch/combine phase contract and the
// kernel launches.
//
// Phase contract (InferenceX PR #2450, "CollectiveX: add FlashInfer
// one-sided NVLink EP for the GB SKUs", "The adapter" table): dispatch
// refuses to run twice without a combine, combine requires a pending
// dispatch, and the state returns to idle after combine;
// runtime_max_tokens_per_rank <= max_num_tokens, with the workspace sized
// once for the maximum.
#include "moe_a2a.h"

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "dispatch_small.h"
#include "expert.h"
#include "kernels.h"

namespace {

// A CUDA call of this library failed.  The status says so; the runtime's
// last error, which a refused launch also leaves behind, is cleared so that
// the caller's next, unrelated CUDA call does not report it again.
int cuda_failed() {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
}

constexpr size_t kAlign = 256;
// Most tokens of a call (all sources) for the cluster combine by default.
// L2-flushed CUDA-event times against the persistent combines (fused,
// H = 7168): 8 tokens 8.2 vs 10.2 us, 64 tokens 10.2 vs 10.2, 256 tokens
// 18.4 vs 12.3, 512 tokens 28.6 vs 18.4: beyond a few dozen tokens its
// CTAs run in waves, each paying the whole chain of round trips, where the
// persistent combines overlap one token's loads with another's epilogue.
constexpr long long kSmallCombineMaxTokens = 64;

// Row tiles per raster group of the expert product by default (each
// weight tile is read from DRAM about once per group).  Measured on the
// moe_layer product (8 experts x 8192 rows, H = N = 7168), full-size DRAM
// bytes per launch and live TFLOP/s: 8 -> 9.83 GB, 1657; 16 -> 6.17 GB, 1761;
// 32 -> 8.08 GB, 1724; 64 -> 13.96 GB, 1581 (the group's rows no longer stay
// in L2 while its weight tiles pass).
constexpr int kGemmGroupM = 16;

int gemm_group_m(const moe::Tuning &tn) {
    return tn.gemm_group_m > 0 ? tn.gemm_group_m : kGemmGroupM;
}

// Largest tokens per rank for the one-launch dispatch by default: one
// routing tile, the most it serves.  Measured faster than the two routing
// passes + row copy at every size up to there (L2 flushed): T = 1 8.9 us,
// T = 64 14.3 vs 18.2-19.1 us, T = 128 20.9 vs 24.5-25.3 us, T = 256
// 33.3-35.2 vs 38.4-38.7 us.
constexpr int kSmallDispatchMaxT = 256;

// Largest tokens per rank for the expert layout's one-launch dispatch by
// default (dispatch_small_expert.cu; each warp reads the ids of every token
// before it, so its work grows with the batch).  Measured faster than the
// two routing passes + row copy at every size up to one routing tile (L2
// flushed, p50): T = 1 8.2 vs 15.8 us, T = 32 12.7 vs 17.8, T = 64 16.8 vs
// 22.0, T = 128 25.0-26.4 vs 30.1, T = 192 35.3 vs 38.3, T = 256 47.6 vs 50.9.
constexpr int kSmallExpertDispatchMaxT = 256;

// The same for the expert layout's FP8 receive rows (one CTA per token):
// faster than the routing passes + FP8 row copy up to 64 tokens per rank
// (p50: T = 1 8.2 vs 13.7 us, T = 32 10.3-12.3 vs 15.8, T = 64 16.3 vs 17.9)
// and slower beyond (T = 128 26.6 vs 24.0, T = 256 53.3 vs 32.2: one CTA per
// token runs in waves).
constexpr int kSmallExpertFp8MaxT = 64;

// The same for FP8 receive rows (one CTA per token, dispatch_small.cu):
// measured faster than the routing passes + FP8 row copy up to 128 tokens
// per rank (T = 1 10.2 vs 14.9 us, T = 64 13.4 vs 16.8, T = 128 16.4 vs
// 21.0) and slower at 256 (30.7 vs 26.5: 2048 CTAs in waves).
constexpr int kSmallFp8MaxT = 128;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t recv_x, expert_out, recv_ids, recv_w, recv_scale, src_token, recv_counts,
        local_counts, local_counts2, recv_counts2;
    size_t send_slot, dest_weight, topk_dest, tile_counts, tile_prefix, tile_ticket, hist_accum,
        local_slot, flags;
    size_t total;
    int layout;      // MOE_LAYOUT_*
    int RP, ntiles_max;
    int P;           // send-row entries per token: RP (rank) or KP (expert)
};

bool config_ok(const moe_a2a_config_t *c) {
    if (c == nullptr) return false;
    if (c->ep_size < 1 || c->ep_size > MOE_MAX_EP_SIZE) return false;
    if (c->max_tokens_per_rank < 1 || c->max_tokens_per_rank > (1 << 24)) return false;
    if (c->hidden < 8 || c->hidden > MOE_MAX_HIDDEN || c->hidden % 8 != 0) return false;
    if (c->num_experts < c->ep_size || c->num_experts > MOE_MAX_EXPERTS) return false;
    if (c->num_experts % c->ep_size != 0) return false;
    if (c->top_k < 1 || c->top_k > MOE_MAX_TOP_K) return false;
    return true;
}

// Regions of the workspace, each 256-byte aligned, sized for M tokens.
bool compute_layout(const moe_a2a_config_t *c, int layout, Layout *L) {
    if (!config_ok(c)) return false;
    if (layout != MOE_LAYOUT_RANK && layout != MOE_LAYOUT_EXPERT) return false;
    const size_t R = c->ep_size, M = c->max_tokens_per_rank, H = c->hidden;
    const size_t E = c->num_experts, K = c->top_k;
    L->layout = layout;
    L->RP = (int)((R + 3) / 4 * 4);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, kAlign);
        return o;
    };
    if (layout == MOE_LAYOUT_EXPERT) {
        // Expert planes of cap = R * M rows; one row per (token, expert).
        if (E > (size_t)moe::kMaxExpertsExpertLayout) return false;
        const size_t KP = (K + 3) / 4 * 4, cap = R * M;
        if (E * cap >= ((size_t)1 << 31)) return false;  // rows are int32 in the send table
        const size_t NT = (M + moe::route_expert_tile() - 1) / moe::route_expert_tile();
        L->P = (int)KP;
        L->ntiles_max = (int)NT;
        L->recv_x = take(E * cap * H * 2);
        L->expert_out = take(E * cap * H * 2);
        L->recv_ids = take(0);
        L->recv_w = take(E * cap * 4);
        L->recv_scale = take(E * cap * 4);
        L->src_token = take(E * cap * 4);
        L->recv_counts = take(E * 4);
        L->local_counts = take(E * 4);
        // the one-launch dispatch alternates two (histogram, rows) pairs
        L->local_counts2 = take(E * 4);
        L->recv_counts2 = take(E * 4);
        L->send_slot = take(R * M * KP * 4);
        L->dest_weight = take(R * M * KP * 4);
        L->topk_dest = take(0);
        L->tile_counts = take(R * NT * E * 4);
        L->tile_prefix = take(0);
        L->tile_ticket = take(0);
        L->hist_accum = take(E * 4);  // zero between calls
        L->local_slot = take(0);
        L->flags = take(kAlign);
        L->total = off;
        return true;
    }
    L->P = L->RP;
    L->ntiles_max = (int)((M + moe::kRouteMinTile - 1) / moe::kRouteMinTile);
    const size_t RP = L->RP, NT = L->ntiles_max;
    L->recv_x = take(R * R * M * H * 2);
    L->expert_out = take(R * R * M * H * 2);
    L->recv_ids = take(R * R * M * K * 4);
    L->recv_w = take(R * R * M * K * 4);
    L->recv_scale = take(R * R * M * 4);
    L->src_token = take(R * R * M * 4);
    L->recv_counts = take(R * R * 4);
    L->local_counts = take(E * 4);
    L->local_counts2 = take(E * 4);  // the one-launch dispatch alternates the two
    L->recv_counts2 = L->recv_counts;  // (its recv counts are written, not added)
    L->send_slot = take(R * M * RP * 4);
    L->dest_weight = take(R * M * RP * 4);
    L->topk_dest = take(R * M * K);
    L->tile_counts = take(R * NT * RP * 4);
    L->tile_prefix = take(R * NT * RP * 4);
    L->tile_ticket = take(R * 4);  // ticket and histogram accumulator are
    L->hist_accum = take(R * E * 4);  // zero between calls
    L->local_slot = take(R * M * RP * 4);
    L->flags = take(kAlign);
    L->total = off;
    return true;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int env_int(const char *name) {
    const char *v = std::getenv(name);
    return (v != nullptr && *v) ? std::atoi(v) : 0;
}

// The tuning switches (kernels.h), read once when a handle is created.
moe::Tuning read_tuning() {
    moe::Tuning tn;
    const char *ov = std::getenv("MOE_ROUTE_OVERLAP");
    tn.route_overlap = (ov != nullptr && ov[0] == '0') ? 0 : 1;
    tn.route_tile = env_int("MOE_ROUTE_TILE");
    tn.dispatch_stages = env_int("MOE_DISPATCH_STAGES");
    tn.dispatch_ctas_per_sm = env_int("MOE_DISPATCH_CTAS_PER_SM");
    tn.fp8_dispatch_stages = env_int("MOE_FP8_DISPATCH_STAGES");
    const char *ck = std::getenv("MOE_COMBINE_KERNEL");
    tn.combine_kernel = ck == nullptr ? 0 : std::strcmp(ck, "ring") == 0 ? 1
                                          : std::strcmp(ck, "regs") == 0 ? 2 : 0;
    tn.combine_ring_slots = env_int("MOE_COMBINE_RING_SLOTS");
    tn.dispatch_small_max = env_int("MOE_DISPATCH_SMALL_MAX");
    tn.gemm_group_m = env_int("MOE_GEMM_GROUP_M");
    tn.combine_small_max = env_int("MOE_COMBINE_SMALL_MAX");
    return tn;
}

}  // namespace

struct moe_a2a {
    moe_a2a_config_t cfg;
    uint8_t *ws;
    size_t ws_bytes;
    Layout L;
    int phase;  // 0 idle, 1 dispatched
    moe::TokenMap map;  // tokens of the pending dispatch
    long long ntok;     // map.first[R]
    int m;              // plane stride of the pending dispatch
    uint32_t active;    // ranks that take part (all by default)
    bool accum_dirty;  // routing pass interrupted: re-zero its accumulators
    int reduction;     // MOE_REDUCE_*
    int recv_format;   // MOE_FORMAT_*
    moe::Tuning tuning;  // read at creation
    // lazily initialised on the first call that queues work
    bool ready;
    int device;
    int num_sms;
    moe::DispatchParams dispatch_tmpl;
    moe::LaunchShape dispatch_shape;
    int fp8_stages;  // FP8 dispatch ring depth and shape (H % 16 == 0 only)
    moe::LaunchShape fp8_shape;
    moe::DispatchSmallShapes small;  // one-launch dispatch (rank layout, or the expert
                                     // layout's own kernel)
    moe::DispatchSmallFp8Shape small_fp8;  // its FP8 receive-row variant
    bool small_fp8_ok;
    int small_fp8_max;  // MOE_DISPATCH_SMALL_FP8_MAX (0: the default, -1: never)
    moe::SmallCombineShape small_combine;  // cluster combine for small batches
    bool small_combine_ok;
    // Local-expert counts: the region holding the current dispatch's counts,
    // and for the one-launch dispatch the buffer (0: local_counts, 1:
    // local_counts2) its next call adds into, and whether that one is zero.
    // The expert layout's one-launch dispatch alternates its rows per expert
    // the same way (recv_counts / recv_counts2, in step with the histogram).
    size_t cur_counts, cur_recv_counts;
    int small_sel;
    bool small_zero_ok;
    // The rank layout's second routing pass runs on `side`, beside the row
    // copy: forked after the first pass (ev_count), joined before the call
    // returns (ev_scan).
    bool overlap;
    cudaStream_t side;
    cudaEvent_t ev_count, ev_scan;
    // combine launch shapes by variant: 4 * out8 + 2 * weighted + fused
    bool combine_ready[8];
    bool combine_ring[8];
    int combine_vpt[8];
    int combine_slots[8];
    moe::LaunchShape combine_shape[8];
};

namespace {

template <typename T>
T *at(moe_a2a_t *h, size_t off) {
    return reinterpret_cast<T *>(h->ws + off);
}

int init_device(moe_a2a_t *h, cudaStream_t st) {
    if (h->ready) return MOE_OK;
    if (cudaGetDevice(&h->device) != cudaSuccess) return cuda_failed();
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
        cudaSuccess)
        return cuda_failed();
    std::memset(&h->dispatch_tmpl, 0, sizeof h->dispatch_tmpl);
    if (moe::dispatch_prepare(2 * h->cfg.hidden, h->L.P, h->num_sms, h->tuning,
                              &h->dispatch_tmpl, &h->dispatch_shape) != cudaSuccess)
        return cuda_failed();
    if (h->cfg.hidden % 16 == 0) {
        moe::DispatchFp8Params fp;
        if (moe::dispatch_fp8_prepare(h->cfg.hidden, h->num_sms, h->tuning, &fp,
                                      &h->fp8_shape) != cudaSuccess)
            return cuda_failed();
        h->fp8_stages = fp.stages;
    }
    if ((h->L.layout == MOE_LAYOUT_RANK
             ? moe::dispatch_small_prepare(2 * h->cfg.hidden, h->num_sms, &h->small)
             : moe::dispatch_small_expert_prepare(2 * h->cfg.hidden, h->num_sms, &h->small)) !=
        cudaSuccess)
        return cuda_failed();
    h->small_fp8_ok =
        h->cfg.hidden % 16 == 0 &&
        (h->L.layout == MOE_LAYOUT_RANK
             ? moe::dispatch_small_fp8_prepare(h->cfg.hidden, &h->small_fp8)
             : moe::dispatch_small_expert_fp8_prepare(h->cfg.hidden, &h->small_fp8)) ==
            cudaSuccess;
    if (cudaMemsetAsync(h->ws + h->L.flags, 0, sizeof(uint32_t), st) != cudaSuccess)
        return cuda_failed();
    h->overlap = h->L.layout == MOE_LAYOUT_RANK && h->tuning.route_overlap != 0;
    h->small_combine_ok = moe::combine_small_shape(h->cfg.hidden, &h->small_combine);
    if (h->overlap) {  // each object once, also after a partial failure
        if (h->side == nullptr &&
            cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess)
            return cuda_failed();
        if (h->ev_count == nullptr &&
            cudaEventCreateWithFlags(&h->ev_count, cudaEventDisableTiming) != cudaSuccess)
            return cuda_failed();
        if (h->ev_scan == nullptr &&
            cudaEventCreateWithFlags(&h->ev_scan, cudaEventDisableTiming) != cudaSuccess)
            return cuda_failed();
    }
    h->accum_dirty = true;  // routing accumulators: zero them before the first pass
    h->ready = true;
    return MOE_OK;
}

// Where the send-table entries of the current call point (kernels.h).
moe::DestRows dest_rows(const moe_a2a_t *h, int m) {
    moe::DestRows D;
    D.P = h->L.P;
    D.expert = h->L.layout == MOE_LAYOUT_EXPERT;
    D.cap = h->cfg.ep_size * m;
    D.rows = (long long)h->cfg.num_experts * D.cap;
    D.Epr = h->cfg.num_experts / h->cfg.ep_size;
    return D;
}

void uniform_map(int R, int T, moe::TokenMap *map) {
    map->stride = T;
    map->uniform = 1;
    for (int s = 0; s < moe::kMaxRanks; ++s) {
        map->count[s] = s < R ? T : 0;
        map->first[s] = (s < R ? s : R) * T;
    }
    map->first[moe::kMaxRanks] = R * T;
}

// The row copy of the dispatch phase (after the routing pass queued its
// send table): bf16 rows, or e4m3 rows + scales in the FP8 receive format.
//
// With `tile` > 0 (rank layout, second routing pass still running) the copy
// reads the first pass's tile-local slots and adds the tile prefixes.
int launch_rows(moe_a2a_t *h, const void *d_x, const moe::TokenMap &map, int m,
                const moe::DestRows &dest, long long ntok, cudaStream_t st, int tile = 0,
                int ntiles = 0) {
    const int R = h->cfg.ep_size;
    uint32_t *flags = at<uint32_t>(h, h->L.flags);
    if (h->recv_format == MOE_FORMAT_FP8_E4M3) {
        moe::DispatchFp8Params fp;
        fp.x = static_cast<const uint16_t *>(d_x);
        fp.send_slot = at<int32_t>(h, h->L.send_slot);
        fp.recv_x8 = at<uint8_t>(h, h->L.recv_x);
        fp.recv_scale = at<float>(h, h->L.recv_scale);
        fp.flags = flags;
        fp.map = map;
        fp.dest = dest;
        fp.R = R, fp.RP = h->L.RP, fp.m = m;
        fp.H = h->cfg.hidden, fp.H8 = h->cfg.hidden / 8;
        fp.tokens = ntok;
        fp.stages = h->fp8_stages;
        fp.tile_prefix = nullptr;
        fp.tile = fp.ntiles = 0;
        if (tile > 0) {
            fp.send_slot = at<int32_t>(h, h->L.local_slot);
            fp.tile_prefix = at<int32_t>(h, h->L.tile_prefix);
            fp.tile = tile, fp.ntiles = ntiles;
        }
        return moe::launch_dispatch_fp8(fp, h->fp8_shape, st) == cudaSuccess ? MOE_OK
                                                                              : cuda_failed();
    }
    moe::DispatchParams dp = h->dispatch_tmpl;
    dp.x = static_cast<const uint8_t *>(d_x);
    dp.send_slot = at<int32_t>(h, h->L.send_slot);
    dp.recv_x = at<uint8_t>(h, h->L.recv_x);
    dp.flags = flags;
    dp.map = map;
    dp.dest = dest;
    dp.R = R, dp.RP = h->L.RP, dp.m = m;
    dp.units = ntok * dp.chunks;
    if (tile > 0) {
        dp.send_slot = at<int32_t>(h, h->L.local_slot);
        dp.tile_prefix = at<int32_t>(h, h->L.tile_prefix);
        dp.tile = tile, dp.ntiles = ntiles;
    }
    return moe::launch_dispatch_rows(dp, h->dispatch_shape, st, true) == cudaSuccess
               ? MOE_OK
               : cuda_failed();
}

// The one-launch dispatch (dispatch_small.cu) serves the rank layout's bf16
// rows when every source holds the same T tokens, T at most one routing tile
// and at most Tuning::dispatch_small_max (measured break-even, below).
bool small_dispatch(const moe_a2a_t *h, const moe::TokenMap &map) {
    if (!map.uniform) return false;
    if (h->L.layout == MOE_LAYOUT_EXPERT) {
        int T_max = 0;
        if (h->recv_format == MOE_FORMAT_BF16) {
            const int lim = h->tuning.dispatch_small_max;
            T_max = lim < 0 ? 0 : (lim == 0 ? kSmallExpertDispatchMaxT : lim);
        } else if (h->recv_format == MOE_FORMAT_FP8_E4M3 && h->small_fp8_ok) {
            const int lim = h->small_fp8_max;
            T_max = lim < 0 ? 0 : (lim == 0 ? kSmallExpertFp8MaxT : lim);
        }
        return map.stride >= 1 && map.stride <= T_max && map.stride <= moe::kRouteTile;
    }
    int T_max = 0;
    if (h->recv_format == MOE_FORMAT_BF16) {
        const int lim = h->tuning.dispatch_small_max;
        T_max = lim < 0 ? 0 : (lim == 0 ? kSmallDispatchMaxT : lim);
    } else if (h->recv_format == MOE_FORMAT_FP8_E4M3 && h->small_fp8_ok) {
        const int lim = h->small_fp8_max;
        T_max = lim < 0 ? 0 : (lim == 0 ? kSmallFp8MaxT : lim);
    }
    return map.stride >= 1 && map.stride <= T_max && map.stride <= moe::kRouteTile;
}

// The cluster combine (combine_small.cu) serves bf16 outputs of calls with
// at most Tuning::combine_small_max tokens (all sources).
bool small_combine(const moe_a2a_t *h, long long ntok) {
    const int lim = h->tuning.combine_small_max;
    const long long most = lim < 0 ? 0 : (lim == 0 ? kSmallCombineMaxTokens : lim);
    return h->small_combine_ok && ntok <= most;
}

// The dispatch phase for the tokens described by `map` (rows of stride
// map.stride in the [R][stride] input arrays).
int dispatch_impl(moe_a2a_t *h, const int32_t *d_topk_ids, const float *d_topk_w,
                  const void *d_x, const moe::TokenMap &map, int m, void *stream,
                  moe_dispatch_view_t *out_view) {
    const int R = h->cfg.ep_size, E = h->cfg.num_experts, K = h->cfg.top_k;
    const long long ntok = map.first[R];
    if (ntok > 0) {
        if (d_topk_ids == nullptr || d_topk_w == nullptr || d_x == nullptr)
            return MOE_ERR_INVALID_ARG;
        if (!aligned(d_topk_ids, 4) || !aligned(d_topk_w, 4) || !aligned(d_x, 16))
            return MOE_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = init_device(h, st);
    if (rc != MOE_OK) return rc;

    const int RP = h->L.RP;
    uint32_t *flags = at<uint32_t>(h, h->L.flags);
    int tmax = 0;
    for (int s = 0; s < R; ++s) tmax = map.count[s] > tmax ? map.count[s] : tmax;

    const bool expert = h->L.layout == MOE_LAYOUT_EXPERT;
    const moe::DestRows dest = dest_rows(h, m);
    // The one-launch dispatch alternates its two local-expert count buffers
    // on the host (each call adds into the one the previous call cleared),
    // which a CUDA graph cannot replay: a captured call would add into the
    // same buffer at every replay.  While `stream` is capturing, the call
    // takes the routing passes, whose accumulators are cleared inside the
    // call.  (An unknown capture state counts as capturing.)
    bool one_launch = ntok > 0 && small_dispatch(h, map);
    if (one_launch) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            one_launch = false;
    }
    if (ntok == 0) {
        const size_t nrc = expert ? (size_t)E : (size_t)R * R;
        if (cudaMemsetAsync(h->ws + h->L.recv_counts, 0, sizeof(int32_t) * nrc, st) !=
                cudaSuccess ||
            cudaMemsetAsync(h->ws + h->L.local_counts, 0, sizeof(int32_t) * E, st) !=
                cudaSuccess)
            return cuda_failed();
    } else if (expert && one_launch) {
        // one launch: every copy warp derives its token's rows itself
        const size_t hist[2] = {h->L.local_counts, h->L.local_counts2};
        const size_t rows[2] = {h->L.recv_counts, h->L.recv_counts2};
        const int sel = h->small_sel;
        if (!h->small_zero_ok &&
            (cudaMemsetAsync(h->ws + hist[sel], 0, sizeof(int32_t) * E, st) != cudaSuccess ||
             cudaMemsetAsync(h->ws + rows[sel], 0, sizeof(int32_t) * E, st) != cudaSuccess))
            return cuda_failed();
        if (h->recv_format == MOE_FORMAT_FP8_E4M3) {  // e4m3 rows, one CTA per token
            moe::DispatchSmallExpertFp8Params fp;
            fp.topk_ids = d_topk_ids;
            fp.topk_w = d_topk_w;
            fp.x = static_cast<const uint16_t *>(d_x);
            fp.recv_x8 = at<uint8_t>(h, h->L.recv_x);
            fp.recv_scale = at<float>(h, h->L.recv_scale);
            fp.send_row = at<int32_t>(h, h->L.send_slot);
            fp.wsum = at<float>(h, h->L.dest_weight);
            fp.src_token = at<int32_t>(h, h->L.src_token);
            fp.recv_w = at<float>(h, h->L.recv_w);
            fp.counts = at<int32_t>(h, hist[sel]);
            fp.counts_clear = at<int32_t>(h, hist[sel ^ 1]);
            fp.recv_counts = at<int32_t>(h, rows[sel]);
            fp.recv_counts_clear = at<int32_t>(h, rows[sel ^ 1]);
            fp.flags = flags;
            fp.active = h->active;
            fp.R = R, fp.K = K, fp.E = E, fp.Epr = E / R, fp.KP = h->L.P, fp.T = map.stride;
            fp.cap = dest.cap, fp.H = h->cfg.hidden, fp.H8 = h->cfg.hidden / 8;
            h->small_zero_ok = false;  // until the launch that clears the other pair is queued
            if (moe::launch_dispatch_small_expert_fp8(fp, h->small_fp8, st) != cudaSuccess)
                return cuda_failed();
        } else {
            const int row_bytes = 2 * h->cfg.hidden;
            const int c = moe::dispatch_small_chunks(row_bytes, h->num_sms, ntok);
            moe::DispatchSmallExpertParams sp;
            sp.topk_ids = d_topk_ids;
            sp.topk_w = d_topk_w;
            sp.x = static_cast<const uint8_t *>(d_x);
            sp.recv_x = at<uint8_t>(h, h->L.recv_x);
            sp.send_row = at<int32_t>(h, h->L.send_slot);
            sp.wsum = at<float>(h, h->L.dest_weight);
            sp.src_token = at<int32_t>(h, h->L.src_token);
            sp.recv_w = at<float>(h, h->L.recv_w);
            sp.counts = at<int32_t>(h, hist[sel]);
            sp.counts_clear = at<int32_t>(h, hist[sel ^ 1]);
            sp.recv_counts = at<int32_t>(h, rows[sel]);
            sp.recv_counts_clear = at<int32_t>(h, rows[sel ^ 1]);
            sp.flags = flags;
            sp.active = h->active;
            sp.R = R, sp.K = K, sp.E = E, sp.Epr = E / R, sp.KP = h->L.P, sp.T = map.stride;
            sp.cap = dest.cap;
            sp.row_bytes = row_bytes;
            sp.chunk_bytes = h->small.chunk_bytes[c];
            sp.chunks = h->small.chunks[c];
            sp.stages = h->small.stages;
            sp.stage_bytes = h->small.stage_bytes[c];
            sp.units = ntok * sp.chunks;
            h->small_zero_ok = false;  // until the launch that clears the other pair is queued
            if (moe::launch_dispatch_small_expert(sp, h->small.shape[c], st) != cudaSuccess)
                return cuda_failed();
        }
        h->cur_counts = hist[sel];
        h->cur_recv_counts = rows[sel];
        h->small_sel = sel ^ 1;
        h->small_zero_ok = true;
    } else if (expert) {
        if (h->accum_dirty) {  // the histogram accumulator
            if (cudaMemsetAsync(h->ws + h->L.hist_accum, 0, sizeof(int32_t) * E, st) !=
                cudaSuccess)
                return cuda_failed();
            h->accum_dirty = false;
        }
        moe::RouteExpertParams rp;
        rp.topk_ids = d_topk_ids;
        rp.topk_w = d_topk_w;
        rp.tile_counts = at<int32_t>(h, h->L.tile_counts);
        rp.send_row = at<int32_t>(h, h->L.send_slot);
        rp.wsum = at<float>(h, h->L.dest_weight);
        rp.src_token = at<int32_t>(h, h->L.src_token);
        rp.recv_w = at<float>(h, h->L.recv_w);
        rp.recv_counts = at<int32_t>(h, h->L.recv_counts);
        rp.hist_accum = at<int32_t>(h, h->L.hist_accum);
        rp.local_counts = at<int32_t>(h, h->L.local_counts);
        rp.flags = flags;
        rp.map = map;
        rp.active = h->active;
        rp.R = R, rp.K = K, rp.E = E, rp.Epr = E / R, rp.KP = h->L.P, rp.cap = dest.cap;
        rp.ntiles = (tmax + moe::route_expert_tile() - 1) / moe::route_expert_tile();
        // Top-k slots per CTA of the second pass: all, or one each while the
        // (tile, source) grid would cover fewer than half the SMs.
        rp.kg = R * rp.ntiles * 2 >= h->num_sms ? rp.KP : 1;
        h->accum_dirty = true;  // until the pass that clears the accumulator is queued
        if (moe::launch_route_expert(rp, st) != cudaSuccess) return cuda_failed();
        h->accum_dirty = false;
        rc = launch_rows(h, d_x, map, m, dest, ntok, st);
        if (rc != MOE_OK) return rc;
    } else if (one_launch) {
        // one launch: every copy warp derives its token's slots itself
        const size_t bufs[2] = {h->L.local_counts, h->L.local_counts2};
        const int sel = h->small_sel;
        if (!h->small_zero_ok &&
            cudaMemsetAsync(h->ws + bufs[sel], 0, sizeof(int32_t) * E, st) != cudaSuccess)
            return cuda_failed();
        const int T = map.stride;
        if (h->recv_format == MOE_FORMAT_FP8_E4M3) {  // e4m3 rows, one CTA per token
            moe::DispatchSmallFp8Params fp;
            fp.topk_ids = d_topk_ids;
            fp.topk_w = d_topk_w;
            fp.x = static_cast<const uint16_t *>(d_x);
            fp.recv_x8 = at<uint8_t>(h, h->L.recv_x);
            fp.recv_scale = at<float>(h, h->L.recv_scale);
            fp.send_slot = at<int32_t>(h, h->L.send_slot);
            fp.dest_weight = at<float>(h, h->L.dest_weight);
            fp.src_token = at<int32_t>(h, h->L.src_token);
            fp.recv_ids = at<int32_t>(h, h->L.recv_ids);
            fp.recv_w = at<float>(h, h->L.recv_w);
            fp.topk_dest = at<int8_t>(h, h->L.topk_dest);
            fp.recv_counts = at<int32_t>(h, h->L.recv_counts);
            fp.counts = at<int32_t>(h, bufs[sel]);
            fp.counts_clear = at<int32_t>(h, bufs[sel ^ 1]);
            fp.flags = flags;
            fp.active = h->active;
            fp.R = R, fp.K = K, fp.E = E, fp.Epr = E / R, fp.RP = RP, fp.m = m, fp.T = T;
            fp.H = h->cfg.hidden, fp.H8 = h->cfg.hidden / 8;
            h->small_zero_ok = false;  // until the launch that clears the other buffer is queued
            if (moe::launch_dispatch_small_fp8(fp, h->small_fp8, st) != cudaSuccess)
                return cuda_failed();
        } else {
            const int row_bytes = 2 * h->cfg.hidden;
            const int c = moe::dispatch_small_chunks(row_bytes, h->num_sms, ntok);
            moe::DispatchSmallParams sp;
            sp.topk_ids = d_topk_ids;
            sp.topk_w = d_topk_w;
            sp.x = static_cast<const uint8_t *>(d_x);
            sp.recv_x = at<uint8_t>(h, h->L.recv_x);
            sp.send_slot = at<int32_t>(h, h->L.send_slot);
            sp.dest_weight = at<float>(h, h->L.dest_weight);
            sp.src_token = at<int32_t>(h, h->L.src_token);
            sp.recv_ids = at<int32_t>(h, h->L.recv_ids);
            sp.recv_w = at<float>(h, h->L.recv_w);
            sp.topk_dest = at<int8_t>(h, h->L.topk_dest);
            sp.recv_counts = at<int32_t>(h, h->L.recv_counts);
            sp.counts = at<int32_t>(h, bufs[sel]);
            sp.counts_clear = at<int32_t>(h, bufs[sel ^ 1]);
            sp.flags = flags;
            sp.active = h->active;
            sp.R = R, sp.K = K, sp.E = E, sp.Epr = E / R, sp.RP = RP, sp.m = m, sp.T = T;
            sp.row_bytes = row_bytes;
            sp.chunk_bytes = h->small.chunk_bytes[c];
            sp.chunks = h->small.chunks[c];
            sp.stages = h->small.stages;
            sp.stage_bytes = h->small.stage_bytes[c];
            sp.units = ntok * sp.chunks;
            h->small_zero_ok = false;  // until the launch that clears the other buffer is queued
            if (moe::launch_dispatch_small(sp, h->small.shape[c], st) != cudaSuccess)
                return cuda_failed();
        }
        h->cur_counts = bufs[sel];
        h->cur_recv_counts = h->L.recv_counts;
        h->small_sel = sel ^ 1;
        h->small_zero_ok = true;
    } else {
        if (h->accum_dirty) {
            if (cudaMemsetAsync(h->ws + h->L.tile_ticket, 0, sizeof(int32_t) * R, st) !=
                    cudaSuccess ||
                cudaMemsetAsync(h->ws + h->L.hist_accum, 0, sizeof(int32_t) * R * E, st) !=
                    cudaSuccess)
                return cuda_failed();
            h->accum_dirty = false;
        }
        const int tile = moe::route_tile(h->tuning);
        const int ntiles = (tmax + tile - 1) / tile;

        moe::RouteCountParams rc_p;
        rc_p.topk_ids = d_topk_ids;
        rc_p.tile_counts = at<int32_t>(h, h->L.tile_counts);
        rc_p.tile_prefix = at<int32_t>(h, h->L.tile_prefix);
        rc_p.tile_ticket = at<int32_t>(h, h->L.tile_ticket);
        rc_p.hist_accum = at<int32_t>(h, h->L.hist_accum);
        rc_p.recv_counts = at<int32_t>(h, h->L.recv_counts);
        rc_p.flags = flags;
        rc_p.map = map;
        rc_p.active = h->active;
        rc_p.R = R, rc_p.K = K, rc_p.E = E, rc_p.Epr = E / R, rc_p.RP = RP;
        rc_p.ntiles = ntiles;
        rc_p.tile = tile;
        const bool overlap = h->overlap;
        rc_p.local_slot = overlap ? at<int32_t>(h, h->L.local_slot) : nullptr;
        if (moe::launch_route_count(rc_p, st) != cudaSuccess) return cuda_failed();
        h->accum_dirty = true;  // until the scan pass that clears it is queued

        moe::RouteScanParams rs;
        rs.topk_ids = d_topk_ids;
        rs.topk_w = d_topk_w;
        rs.tile_prefix = rc_p.tile_prefix;
        rs.hist_accum = rc_p.hist_accum;
        rs.send_slot = at<int32_t>(h, h->L.send_slot);
        rs.dest_weight = at<float>(h, h->L.dest_weight);
        rs.src_token = at<int32_t>(h, h->L.src_token);
        rs.recv_ids = at<int32_t>(h, h->L.recv_ids);
        rs.recv_w = at<float>(h, h->L.recv_w);
        rs.topk_dest = at<int8_t>(h, h->L.topk_dest);
        rs.local_counts = at<int32_t>(h, h->L.local_counts);
        rs.map = map;
        rs.active = h->active;
        rs.R = R, rs.K = K, rs.E = E, rs.Epr = E / R, rs.RP = RP, rs.m = m;
        rs.ntiles = ntiles;
        rs.tile = tile;
        // Destinations per CTA of the second pass: 4 (16-byte send-row
        // stores) once the grid has a CTA per SM, else 1 so that a small
        // batch's per-destination work spreads over RP times the CTAs.
        rs.dg = R * ntiles * (RP / 4) >= h->num_sms ? 4 : 1;
        if (overlap) {
            // The row copy needs only the first pass; the second (send
            // table, weights, metadata rows) runs beside it on `side`.
            if (cudaEventRecord(h->ev_count, st) != cudaSuccess ||
                cudaStreamWaitEvent(h->side, h->ev_count, 0) != cudaSuccess)
                return cuda_failed();
            if (moe::launch_route_scan(rs, h->side, false) != cudaSuccess) return cuda_failed();
            const int rows_rc = launch_rows(h, d_x, map, m, dest, ntok, st, tile, ntiles);
            // Join whatever happened to the copy, so `side` never outlives the call.
            if (cudaEventRecord(h->ev_scan, h->side) != cudaSuccess ||
                cudaStreamWaitEvent(st, h->ev_scan, 0) != cudaSuccess)
                return cuda_failed();
            h->accum_dirty = false;
            if (rows_rc != MOE_OK) return rows_rc;
        } else {
            if (moe::launch_route_scan(rs, st, true) != cudaSuccess) return cuda_failed();
            h->accum_dirty = false;
            rc = launch_rows(h, d_x, map, m, dest, ntok, st);
            if (rc != MOE_OK) return rc;
        }
    }

    if (!one_launch) {
        // the routing pass (or the empty call) wrote local_counts and
        // recv_counts (the first buffer of each pair)
        h->cur_counts = h->L.local_counts;
        h->cur_recv_counts = h->L.recv_counts;
        if (h->small_sel == 0) h->small_zero_ok = false;
    }
    h->map = map;
    h->ntok = ntok;
    h->m = m;
    h->phase = 1;
    if (out_view != nullptr) {
        out_view->recv_x = h->ws + h->L.recv_x;
        out_view->recv_topk_ids = expert ? nullptr : at<int32_t>(h, h->L.recv_ids);
        out_view->recv_topk_w = at<float>(h, h->L.recv_w);
        out_view->src_token = at<int32_t>(h, h->L.src_token);
        out_view->recv_counts = at<int32_t>(h, h->cur_recv_counts);
        out_view->local_expert_counts = at<int32_t>(h, h->cur_counts);
        out_view->send_slot = at<int32_t>(h, h->L.send_slot);
        out_view->dest_weight = at<float>(h, h->L.dest_weight);
        out_view->plane_stride = expert ? dest.cap : m;
        out_view->tokens_per_rank = map.uniform ? map.stride : -1;
        out_view->send_stride = h->L.P;
        out_view->token_stride = map.stride;
        const bool fp8 = h->recv_format == MOE_FORMAT_FP8_E4M3;
        out_view->recv_scale = fp8 ? at<float>(h, h->L.recv_scale) : nullptr;
        out_view->recv_format = h->recv_format;
        out_view->layout = h->L.layout;
        // route_count + route_scan (or the expert layout's two passes) + the
        // row copy, or the one-launch dispatch
        out_view->kernels = ntok == 0 ? 0 : (one_launch ? 1 : 3);
    }
    return MOE_OK;
}

// The combine phase; out8 selects the FP8 output (d_out = e4m3 rows plus
// d_out_scale) instead of bf16 rows.
int combine_impl(moe_a2a_t *h, const void *d_expert_out, int32_t weighted, const void *d_residual,
                 const void *d_gamma, float eps, void *d_out, float *d_out_scale,
                 void *d_residual_out, bool out8, void *stream) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 1) return MOE_ERR_PHASE;
    const bool fused = d_residual != nullptr;
    const void *eo = d_expert_out != nullptr ? d_expert_out : h->ws + h->L.expert_out;
    if (h->ntok > 0) {
        if (d_out == nullptr || !aligned(d_out, 16) || !aligned(eo, 16))
            return MOE_ERR_INVALID_ARG;
        if (out8 && (d_out_scale == nullptr || !aligned(d_out_scale, 4)))
            return MOE_ERR_INVALID_ARG;
        if (fused && (d_gamma == nullptr || !aligned(d_residual, 16) || !aligned(d_gamma, 16)))
            return MOE_ERR_INVALID_ARG;
        if (fused && d_residual_out != nullptr && !aligned(d_residual_out, 16))
            return MOE_ERR_INVALID_ARG;
        if (!fused && d_residual_out != nullptr) return MOE_ERR_INVALID_ARG;
        if (!(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    }
    if (h->reduction == MOE_REDUCE_BF16_TOPK_TREE && (weighted || out8))
        return MOE_ERR_INVALID_ARG;  // (the tree exists for the rank layout only)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (h->ntok > 0 && h->reduction == MOE_REDUCE_BF16_TOPK_TREE) {
        moe::CombineTreeParams tp;
        tp.expert_out = static_cast<const uint16_t *>(eo);
        tp.send_slot = at<int32_t>(h, h->L.send_slot);
        tp.topk_dest = at<int8_t>(h, h->L.topk_dest);
        tp.residual = static_cast<const uint16_t *>(d_residual);
        tp.gamma = static_cast<const uint16_t *>(d_gamma);
        tp.out = static_cast<uint16_t *>(d_out);
        tp.residual_out = static_cast<uint16_t *>(d_residual_out);
        tp.flags = at<uint32_t>(h, h->L.flags);
        tp.eps = eps;
        tp.map = h->map;
        tp.active = h->active;
        tp.R = h->cfg.ep_size, tp.RP = h->L.RP, tp.m = h->m;
        tp.H = h->cfg.hidden, tp.H8 = h->cfg.hidden / 8, tp.K = h->cfg.top_k;
        tp.P = 1;
        while (tp.P < tp.K) tp.P *= 2;
        tp.tokens = h->ntok;
        if (moe::launch_combine_tree(tp, h->num_sms, st) != cudaSuccess) return cuda_failed();
    } else if (h->ntok > 0 && !out8 && small_combine(h, h->ntok)) {
        // few tokens: each row split over a cluster, all its messages in flight
        moe::CombineParams cp;
        cp.expert_out = static_cast<const uint16_t *>(eo);
        cp.send_slot = at<int32_t>(h, h->L.send_slot);
        cp.dest_weight = at<float>(h, h->L.dest_weight);
        cp.residual = static_cast<const uint16_t *>(d_residual);
        cp.gamma = static_cast<const uint16_t *>(d_gamma);
        cp.out = static_cast<uint16_t *>(d_out);
        cp.residual_out = static_cast<uint16_t *>(d_residual_out);
        cp.out8 = nullptr;
        cp.out_scale = nullptr;
        cp.eps = eps;
        cp.flags = at<uint32_t>(h, h->L.flags);
        cp.map = h->map;
        cp.active = h->active;
        cp.dest = dest_rows(h, h->m);
        cp.R = h->cfg.ep_size, cp.RP = h->L.RP, cp.m = h->m;
        cp.H = h->cfg.hidden, cp.H8 = h->cfg.hidden / 8;
        cp.tokens = h->ntok;
        cp.ring_slots = 0;
        if (moe::launch_combine_small(cp, weighted != 0, fused, h->small_combine, st) !=
            cudaSuccess)
            return cuda_failed();
    } else if (h->ntok > 0) {
        const int variant = (out8 ? 4 : 0) + (weighted ? 2 : 0) + (fused ? 1 : 0);
        if (!h->combine_ready[variant]) {
            // Every combine streams its rows through a shared-memory ring
            // (the fused epilogue then overlaps other tokens' loads; the
            // plain sum keeps more rows in flight than registers allow:
            // wide EP 163.6 us against 166.6-167.7 us for the register
            // combine).  Tuning::combine_kernel overrides ("regs": the
            // register combine where it exists; the FP8 output exists on
            // the ring kernel only).
            bool ring = true;
            if (h->tuning.combine_kernel == 2) ring = out8;
            if (h->tuning.combine_kernel == 1) ring = true;
            cudaError_t e =
                ring ? moe::combine_ring_prepare(h->cfg.hidden, weighted != 0, fused, out8,
                                                 h->num_sms, h->tuning,
                                                 &h->combine_shape[variant],
                                                 &h->combine_vpt[variant],
                                                 &h->combine_slots[variant])
                     : moe::combine_prepare(h->cfg.hidden, weighted != 0, fused, h->num_sms,
                                            &h->combine_shape[variant], &h->combine_vpt[variant]);
            if (e != cudaSuccess) return cuda_failed();
            h->combine_ring[variant] = ring;
            h->combine_ready[variant] = true;
        }
        moe::CombineParams cp;
        cp.expert_out = static_cast<const uint16_t *>(eo);
        cp.send_slot = at<int32_t>(h, h->L.send_slot);
        cp.dest_weight = at<float>(h, h->L.dest_weight);
        cp.residual = static_cast<const uint16_t *>(d_residual);
        cp.gamma = static_cast<const uint16_t *>(d_gamma);
        cp.out = out8 ? nullptr : static_cast<uint16_t *>(d_out);
        cp.residual_out = static_cast<uint16_t *>(d_residual_out);
        cp.out8 = out8 ? static_cast<uint8_t *>(d_out) : nullptr;
        cp.out_scale = out8 ? d_out_scale : nullptr;
        cp.eps = eps;
        cp.flags = at<uint32_t>(h, h->L.flags);
        cp.map = h->map;
        cp.active = h->active;
        cp.dest = dest_rows(h, h->m);
        cp.R = h->cfg.ep_size, cp.RP = h->L.RP, cp.m = h->m;
        cp.H = h->cfg.hidden, cp.H8 = h->cfg.hidden / 8;
        cp.tokens = h->ntok;
        cp.ring_slots = h->combine_slots[variant];
        const cudaError_t e =
            h->combine_ring[variant]
                ? moe::launch_combine_ring(cp, weighted != 0, fused, out8,
                                           h->combine_vpt[variant], h->combine_shape[variant], st)
                : moe::launch_combine(cp, weighted != 0, fused, h->combine_vpt[variant],
                                      h->combine_shape[variant], st);
        if (e != cudaSuccess) return cuda_failed();
    }
    h->phase = 0;
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_a2a_workspace_bytes(const moe_a2a_config_t *cfg) {
    return moe_a2a_workspace_bytes_layout(cfg, MOE_LAYOUT_RANK);
}

size_t moe_a2a_workspace_bytes_layout(const moe_a2a_config_t *cfg, int32_t layout) {
    Layout L;
    return compute_layout(cfg, layout, &L) ? L.total : 0;
}

int moe_a2a_create(const moe_a2a_config_t *cfg, void *d_workspace, size_t workspace_bytes,
                   moe_a2a_t **out) {
    return moe_a2a_create_layout(cfg, MOE_LAYOUT_RANK, d_workspace, workspace_bytes, out);
}

int moe_a2a_create_layout(const moe_a2a_config_t *cfg, int32_t layout, void *d_workspace,
                          size_t workspace_bytes, moe_a2a_t **out) {
    if (out == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    Layout L;
    if (!compute_layout(cfg, layout, &L)) return MOE_ERR_INVALID_ARG;
    if (d_workspace == nullptr || !aligned(d_workspace, kAlign)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return MOE_ERR_CAPACITY;
    moe_a2a_t *h = new (std::nothrow) moe_a2a_t;
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    std::memset(h, 0, sizeof *h);
    h->cfg = *cfg;
    h->ws = static_cast<uint8_t *>(d_workspace);
    h->ws_bytes = workspace_bytes;
    h->L = L;
    h->phase = 0;
    h->active = cfg->ep_size >= 32 ? 0xffffffffu : ((1u << cfg->ep_size) - 1u);
    h->tuning = read_tuning();
    h->small_fp8_max = env_int("MOE_DISPATCH_SMALL_FP8_MAX");
    h->small_fp8_ok = false;
    *out = h;
    return MOE_OK;
}

int moe_dispatch(moe_a2a_t *h, const int32_t *d_topk_ids, const float *d_topk_w,
                 const void *d_x, int32_t tokens_per_rank, int32_t runtime_max_tokens_per_rank,
                 void *stream, moe_dispatch_view_t *out_view) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 0) return MOE_ERR_PHASE;
    const int T = tokens_per_rank, m = runtime_max_tokens_per_rank;
    if (T < 0 || m < 1) return MOE_ERR_INVALID_ARG;
    if (m > h->cfg.max_tokens_per_rank || T > m) return MOE_ERR_CAPACITY;
    moe::TokenMap map;
    uniform_map(h->cfg.ep_size, T, &map);
    return dispatch_impl(h, d_topk_ids, d_topk_w, d_x, map, m, stream, out_view);
}

int moe_dispatch_varlen(moe_a2a_t *h, const int32_t *d_topk_ids, const float *d_topk_w,
                        const void *d_x, const int32_t *tokens_per_rank,
                        int32_t runtime_max_tokens_per_rank, void *stream,
                        moe_dispatch_view_t *out_view) {
    if (h == nullptr || tokens_per_rank == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 0) return MOE_ERR_PHASE;
    const int R = h->cfg.ep_size, m = runtime_max_tokens_per_rank;
    if (m < 1) return MOE_ERR_INVALID_ARG;
    if (m > h->cfg.max_tokens_per_rank) return MOE_ERR_CAPACITY;
    moe::TokenMap map;
    map.stride = m;
    map.first[0] = 0;
    bool same = true;
    for (int s = 0; s < R; ++s) {
        const int c = tokens_per_rank[s];
        if (c < 0) return MOE_ERR_INVALID_ARG;
        if (c > m) return MOE_ERR_CAPACITY;
        map.count[s] = c;
        map.first[s + 1] = map.first[s] + c;
        same = same && c == m;
    }
    for (int s = R; s < moe::kMaxRanks; ++s) map.count[s] = 0, map.first[s + 1] = map.first[R];
    map.uniform = same ? 1 : 0;
    return dispatch_impl(h, d_topk_ids, d_topk_w, d_x, map, m, stream, out_view);
}

int moe_a2a_set_active_ranks(moe_a2a_t *h, uint32_t active) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    const uint32_t all =
        h->cfg.ep_size >= 32 ? 0xffffffffu : ((1u << h->cfg.ep_size) - 1u);
    if (active & ~all) return MOE_ERR_INVALID_ARG;
    h->active = active;
    return MOE_OK;
}

void *moe_combine_payload(moe_a2a_t *h) {
    return h == nullptr ? nullptr : h->ws + h->L.expert_out;
}

int moe_combine(moe_a2a_t *h, const void *d_expert_out, int32_t weighted, const void *d_residual,
                const void *d_gamma, float eps, void *d_out, void *d_residual_out, void *stream) {
    return combine_impl(h, d_expert_out, weighted, d_residual, d_gamma, eps, d_out, nullptr,
                        d_residual_out, false, stream);
}

int moe_combine_fp8(moe_a2a_t *h, const void *d_expert_out, int32_t weighted,
                    const void *d_residual, const void *d_gamma, float eps, void *d_out_fp8,
                    float *d_out_scale, void *d_residual_out, void *stream) {
    return combine_impl(h, d_expert_out, weighted, d_residual, d_gamma, eps, d_out_fp8,
                        d_out_scale, d_residual_out, true, stream);
}

int moe_a2a_get_error(moe_a2a_t *h, void *stream, uint32_t *flags) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (flags != nullptr) *flags = 0;
    if (!h->ready) return MOE_OK;  // nothing was ever queued
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, h->ws + h->L.flags, sizeof bits, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return cuda_failed();
    if (bits != 0 &&
        (cudaMemsetAsync(h->ws + h->L.flags, 0, sizeof bits, st) != cudaSuccess ||
         cudaStreamSynchronize(st) != cudaSuccess))
        return cuda_failed();
    if (flags != nullptr) *flags = bits;
    if (bits & MOE_DEVICE_FLAG_WAIT_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    if (bits & MOE_DEVICE_FLAG_BAD_SLOT) return MOE_ERR_INTERNAL;
    if (bits & MOE_DEVICE_FLAG_BAD_EXPERT_ID) return MOE_ERR_ROUTING;
    return MOE_OK;
}

int moe_a2a_destroy(moe_a2a_t *h) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    // Pending work on `side` completes before its resources are released.
    if (h->ev_scan != nullptr) cudaEventDestroy(h->ev_scan);
    if (h->ev_count != nullptr) cudaEventDestroy(h->ev_count);
    if (h->side != nullptr) cudaStreamDestroy(h->side);
    delete h;
    return MOE_OK;
}

int moe_a2a_phase(const moe_a2a_t *h) { return h == nullptr ? -1 : h->phase; }

int moe_a2a_set_recv_format(moe_a2a_t *h, int32_t format) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 0) return MOE_ERR_PHASE;
    if (format == MOE_FORMAT_BF16 || (format == MOE_FORMAT_FP8_E4M3 && h->cfg.hidden % 16 == 0)) {
        h->recv_format = format;
        return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

int moe_quantize_rows_fp8(const float *d_x, int64_t rows, int32_t hidden, void *d_q,
                          float *d_scale, void *stream) {
    if (rows < 0 || hidden < 8 || hidden > MOE_MAX_HIDDEN || hidden % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (d_x == nullptr || d_q == nullptr || d_scale == nullptr || !aligned(d_x, 16) ||
        !aligned(d_q, 16) || !aligned(d_scale, 4))
        return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cuda_failed();
    return moe::launch_quantize_rows_fp8(d_x, rows, hidden, static_cast<uint8_t *>(d_q), d_scale,
                                         sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK
               : cuda_failed();
}

namespace {

int expert_gemm_impl(moe_a2a_t *h, const void *d_w, const float *d_w_scale, int32_t N,
                     void *d_out, bool fp8, void *stream) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 1) return MOE_ERR_PHASE;
    const int H = h->cfg.hidden;
    const int want = fp8 ? MOE_FORMAT_FP8_E4M3 : MOE_FORMAT_BF16;
    if (h->L.layout != MOE_LAYOUT_EXPERT || h->recv_format != want) return MOE_ERR_INVALID_ARG;
    if (H % (fp8 ? 128 : 64) != 0 || N < 128 || N % 128 != 0 || d_w == nullptr ||
        !aligned(d_w, 16))
        return MOE_ERR_INVALID_ARG;
    if (fp8 && (d_w_scale == nullptr || !aligned(d_w_scale, 4))) return MOE_ERR_INVALID_ARG;
    if (d_out == nullptr && N != H) return MOE_ERR_INVALID_ARG;
    if (d_out != nullptr && !aligned(d_out, 16)) return MOE_ERR_INVALID_ARG;
    if (h->ntok == 0) return MOE_OK;
    moe::ExpertGemmParams gp;
    gp.x = h->ws + h->L.recv_x;
    gp.w = d_w;
    gp.out = d_out != nullptr ? d_out : h->ws + h->L.expert_out;
    gp.recv_counts = at<int32_t>(h, h->cur_recv_counts);
    gp.x_scale = fp8 ? at<float>(h, h->L.recv_scale) : nullptr;
    gp.w_scale = fp8 ? d_w_scale : nullptr;
    gp.flags = at<uint32_t>(h, h->L.flags);
    gp.E = h->cfg.num_experts;
    gp.cap = h->cfg.ep_size * h->m;
    gp.H = H;
    gp.N = N;
    gp.mtiles = (gp.cap + 127) / 128;
    gp.fp8 = fp8 ? 1 : 0;
    gp.gather = 0;
    gp.pair_row = nullptr;
    gp.pair_gate = nullptr;
    gp.final_out = nullptr;
    gp.a_rows = 0;
    gp.group_m = gemm_group_m(h->tuning);
    return moe::launch_expert_gemm(gp, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK
               : cuda_failed();
}

// Scratch of the rank-plane product, sized for max_tokens_per_rank: the
// per-expert pair cursors (and the count of rows with several local
// experts), the receive row and gate mark of each pair, the pair of each
// (row, k), the list of rows with several local experts and the experts'
// bf16 outputs, pair-major.
struct RankScratch {
    size_t cursor, pair_row, pair_gate, pair_of, multi, y, total;
    long long multi_cap;
};

bool rank_scratch_layout(const moe_a2a_config_t *c, int N, RankScratch *S) {
    if (!config_ok(c) || N < 128 || N % 128 != 0) return false;
    const size_t R = c->ep_size, M = c->max_tokens_per_rank, K = c->top_k, E = c->num_experts;
    const size_t pairs = R * M * K;  // every token's K ids valid and local somewhere
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, kAlign);
        return o;
    };
    S->cursor = take((E + 1) * 4);  // + the count of rows with several local experts
    S->pair_row = take(pairs * 4);
    S->pair_gate = take(pairs * 4);
    S->pair_of = take(R * R * M * K * 4);
    // such a row holds at least two of the pairs
    S->multi_cap = (long long)(R * M * (K / 2));
    S->multi = take((size_t)S->multi_cap * 4);
    S->y = take(pairs * (size_t)N * 2);
    S->total = off;
    return true;
}

}  // namespace

size_t moe_expert_gemm_rank_scratch_bytes(const moe_a2a_config_t *cfg, int32_t N) {
    RankScratch S;
    return rank_scratch_layout(cfg, N, &S) ? S.total : 0;
}

namespace {

int expert_gemm_rank_impl(moe_a2a_t *h, const void *d_w, const float *d_w_scale, int32_t N,
                          int32_t apply_gates, void *d_out, void *d_scratch,
                          size_t scratch_bytes, bool fp8, void *stream) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->phase != 1) return MOE_ERR_PHASE;
    const int H = h->cfg.hidden, E = h->cfg.num_experts, R = h->cfg.ep_size, K = h->cfg.top_k;
    const int want = fp8 ? MOE_FORMAT_FP8_E4M3 : MOE_FORMAT_BF16;
    if (h->L.layout != MOE_LAYOUT_RANK || h->recv_format != want ||
        E > moe::kMaxExpertsExpertLayout)
        return MOE_ERR_INVALID_ARG;
    if (H % (fp8 ? 128 : 64) != 0 || N < 128 || N % 128 != 0 || d_w == nullptr ||
        !aligned(d_w, 16))
        return MOE_ERR_INVALID_ARG;
    if (fp8 && (d_w_scale == nullptr || !aligned(d_w_scale, 4))) return MOE_ERR_INVALID_ARG;
    if (d_out == nullptr && N != H) return MOE_ERR_INVALID_ARG;
    if (d_out != nullptr && !aligned(d_out, 16)) return MOE_ERR_INVALID_ARG;
    if (d_scratch == nullptr || !aligned(d_scratch, kAlign)) return MOE_ERR_INVALID_ARG;
    if ((long long)R * R * h->m >= (1LL << 31)) return MOE_ERR_INVALID_ARG;  // 31-bit rows
    RankScratch S;
    if (!rank_scratch_layout(&h->cfg, N, &S)) return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < S.total) return MOE_ERR_CAPACITY;
    if (h->ntok == 0) return MOE_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *sc = static_cast<uint8_t *>(d_scratch);
    const int m = h->m;

    moe::RankPairsParams rp;
    rp.recv_ids = at<int32_t>(h, h->L.recv_ids);
    rp.recv_w = at<float>(h, h->L.recv_w);
    rp.recv_counts = at<int32_t>(h, h->cur_recv_counts);
    rp.pair_counts = at<int32_t>(h, h->cur_counts);
    rp.cursor = reinterpret_cast<int32_t *>(sc + S.cursor);
    rp.pair_row = reinterpret_cast<int32_t *>(sc + S.pair_row);
    rp.pair_gate = reinterpret_cast<float *>(sc + S.pair_gate);
    rp.pair_of = reinterpret_cast<int32_t *>(sc + S.pair_of);
    rp.multi = reinterpret_cast<int32_t *>(sc + S.multi);
    rp.multi_cap = S.multi_cap;
    rp.y = reinterpret_cast<const uint16_t *>(sc + S.y);
    rp.out = static_cast<uint16_t *>(d_out != nullptr ? d_out : h->ws + h->L.expert_out);
    rp.flags = at<uint32_t>(h, h->L.flags);
    rp.R = R, rp.m = m, rp.K = K, rp.E = E, rp.N = N;
    rp.apply_gates = apply_gates ? 1 : 0;
    if (cudaMemsetAsync(rp.cursor, 0, sizeof(int32_t) * (E + 1), st) != cudaSuccess)
        return cuda_failed();
    if (moe::launch_rank_pairs(rp, h->num_sms, st) != cudaSuccess) return cuda_failed();

    moe::ExpertGemmParams gp;
    gp.x = h->ws + h->L.recv_x;
    gp.w = d_w;
    gp.out = sc + S.y;
    gp.recv_counts = rp.pair_counts;
    gp.x_scale = fp8 ? at<float>(h, h->L.recv_scale) : nullptr;  // [R][R][m]: per receive row
    gp.w_scale = fp8 ? d_w_scale : nullptr;
    gp.flags = at<uint32_t>(h, h->L.flags);
    gp.E = E;
    gp.cap = R * m * K;  // pairs of one expert at most
    gp.H = H;
    gp.N = N;
    gp.mtiles = (gp.cap + 127) / 128;
    gp.fp8 = fp8 ? 1 : 0;
    gp.gather = 1;
    gp.pair_row = rp.pair_row;
    gp.pair_gate = rp.pair_gate;
    gp.final_out = rp.out;
    gp.a_rows = (long long)R * R * m;
    gp.group_m = gemm_group_m(h->tuning);
    if (moe::launch_expert_gemm(gp, st) != cudaSuccess) return cuda_failed();
    return moe::launch_rank_aggregate(rp, h->num_sms, st) == cudaSuccess ? MOE_OK : cuda_failed();
}

}  // namespace

int moe_expert_gemm_rank(moe_a2a_t *h, const void *d_w, int32_t N, int32_t apply_gates,
                         void *d_out, void *d_scratch, size_t scratch_bytes, void *stream) {
    return expert_gemm_rank_impl(h, d_w, nullptr, N, apply_gates, d_out, d_scratch,
                                 scratch_bytes, false, stream);
}

int moe_expert_gemm_rank_fp8(moe_a2a_t *h, const void *d_w8, const float *d_w_scale, int32_t N,
                             int32_t apply_gates, void *d_out, void *d_scratch,
                             size_t scratch_bytes, void *stream) {
    return expert_gemm_rank_impl(h, d_w8, d_w_scale, N, apply_gates, d_out, d_scratch,
                                 scratch_bytes, true, stream);
}

int moe_expert_gemm(moe_a2a_t *h, const void *d_w, int32_t N, void *d_out, void *stream) {
    return expert_gemm_impl(h, d_w, nullptr, N, d_out, false, stream);
}

int moe_expert_gemm_fp8(moe_a2a_t *h, const void *d_w8, const float *d_w_scale, int32_t N,
                        void *d_out, void *stream) {
    return expert_gemm_impl(h, d_w8, d_w_scale, N, d_out, true, stream);
}

int moe_a2a_set_reduction(moe_a2a_t *h, int32_t reduction) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (reduction == MOE_REDUCE_FP32_RANK_ORDER) {
        h->reduction = reduction;
        return MOE_OK;
    }
    if (reduction == MOE_REDUCE_BF16_TOPK_TREE && h->cfg.top_k <= 8 &&
        h->L.layout == MOE_LAYOUT_RANK) {
        h->reduction = reduction;
        return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

const char *moe_a2a_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_PHASE: return "phase error (dispatch twice, or combine without dispatch)";
        case MOE_ERR_CAPACITY: return "capacity exceeded (runtime max or tokens per rank)";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_ROUTING: return "expert id outside [-1, num_experts) seen on device";
        case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_INTERNAL: return "internal consistency guard fired on device";
        case MOE_ERR_SETUP_IN_CAPTURE:
            return "first allocation-free routing call in a context made during stream capture";
        default: return "unknown status";
    }
}

}  // extern "C"
