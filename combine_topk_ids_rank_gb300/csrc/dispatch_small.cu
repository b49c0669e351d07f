// dispatch_small.cu -- the whole dispatch phase in one launch, for batches
// of at most one routing tile (256 tokens) per source rank.
//
// Operation: the same as route.cu + dispatch.cu (InferenceX PR #2450,
// "CollectiveX: add FlashInfer one-sided NVLink EP for the GB SKUs": "Why",
// "The adapter", the bring-up run table, "Synthesis"):
//   slot(s,t,d) = #{t' < t : d in dmask(s,t')},
//   recv_x[d][s][slot][:] = x[s][t][:] for every d in dmask(s,t),
// with the send table, per-destination weights, source map, masked metadata
// rows, recv counts and local-expert counts of the routing pass.
//
// GB300 design, for small batches where launches and dependent round trips
// cost more than the bytes: one-warp CTAs, several per SM, each taking
// units (a token row, or a chunk of it when there are few tokens) of the
// grid-strided unit list.  A warp derives its token's slots itself from the
// expert ids of the tokens before it in the same source (one warp ballot per
// destination and 32 tokens; at most 8 x 32 tokens), so no CTA waits for
// another and there is no second pass, second stream or event.  Meanwhile
// lane 0 has already requested the unit's x chunk into a shared-memory stage
// with a bulk copy; once the slots are known it stores the chunk to every
// destination row with bulk shared -> global copies.  The warp holding a
// token's first chunk writes its send row, weights, source-map entries and
// metadata rows (the token's ids and weights held one per lane) and adds its
// ids to the local-expert counts with atomics; the warp of a source's last
// token writes its recv counts.  The counts live in one of two buffers that
// alternate between calls: each call adds into the buffer the previous call
// cleared and clears the other one, so nothing waits for a last CTA.
// Waits are bounded: on time-out the kernel raises the flag, drains its
// copies and returns.
#include "dispatch_small.h"
#include "fp8.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "smem_limit.h"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStages = 2;  // x chunks in flight per CTA (shared-memory stages)
constexpr int kSmallFp8MaxThreads = 256;  // threads of the FP8 kernel: at most
constexpr int kMaxTileWords = kRouteTile / 32;  // 32-token groups of a source

// (magic: owner_magic(Epr), kernels.h)
__device__ __forceinline__ int live_rank(int e, int E, unsigned long long magic,
                                         uint32_t active) {
    if (e < 0 || e >= E) return -1;
    const int d = owner_of(e, magic);
    return ((active >> d) & 1u) ? d : -1;
}

// Destination mask of a token: ranks of its valid ids on active ranks.
template <int KT>
__device__ __forceinline__ uint32_t token_mask(const int32_t *ids, int K, int E,
                                               unsigned long long magic, uint32_t active) {
    uint32_t mask = 0;
    if constexpr (KT > 0) {
        int e[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) e[k] = __ldg(ids + k);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int d = live_rank(e[k], E, magic, active);
            if (d >= 0) mask |= 1u << d;
        }
    } else {
        for (int k = 0; k < K; ++k) {
            const int d = live_rank(__ldg(ids + k), E, magic, active);
            if (d >= 0) mask |= 1u << d;
        }
    }
    return mask;
}

// Slots of token t of a source whose ids start at src_ids (one warp): lane d
// gets the number of the source's earlier tokens sent to rank d (cnt), every
// lane the token's destination mask (own).  One ballot per destination and
// 32 earlier tokens.
template <int KT>
__device__ __forceinline__ void token_slots(const int32_t *src_ids, int t, int K, int E, int R,
                                            unsigned long long magic, uint32_t active,
                                            int lane, int &cnt, uint32_t &own) {
    uint32_t masks[kMaxTileWords];
    const int words = t / 32 + 1;
#pragma unroll
    for (int j = 0; j < kMaxTileWords; ++j) masks[j] = 0u;
#pragma unroll
    for (int j = 0; j < kMaxTileWords; ++j) {  // only the words up to token t
        if (j >= words) break;
        const int tt = j * 32 + lane;
        if (tt <= t) masks[j] = token_mask<KT>(src_ids + (size_t)tt * K, K, E, magic, active);
    }
    cnt = 0;
    own = 0;
#pragma unroll
    for (int j = 0; j < kMaxTileWords; ++j) {
        if (j >= words) break;
        const int tt = j * 32 + lane;
        const uint32_t before = tt < t ? masks[j] : 0u;
        for (int d = 0; d < R; ++d) {
            const uint32_t b = __ballot_sync(kFull, (before >> d) & 1u);
            if (lane == d) cnt += __popc(b);
        }
        if (j == t / 32) own = __shfl_sync(kFull, masks[j], t & 31);
    }
}

// The routing outputs of token tok = (s, t) (one warp; its ids and weights
// one per lane): send row and per-destination weights, the top-k slots'
// destinations, the local-expert counts, the source map and metadata rows
// of every destination, and, for the source's last token, its recv counts.
template <class P>
__device__ __forceinline__ void write_routing(const P &p, int K, int tok, int s, int t,
                                              int my_e, float my_w, int cnt, uint32_t own,
                                              int lane) {
    const int my_d = live_rank(my_e, p.E, p.epr_magic, p.active);
    // lane d: the weight sum of the token's experts on d, ascending k from
    // +0.0; lane k: whether slot k is its rank's first
    float wsum = 0.0f;
    bool first_of_rank = my_d >= 0;
    for (int k = 0; k < K; ++k) {
        const int e = __shfl_sync(kFull, my_e, k);
        const float wk = __shfl_sync(kFull, my_w, k);
        const int d = live_rank(e, p.E, p.epr_magic, p.active);
        if (d == lane) wsum = __fadd_rn(wsum, wk);
        if (k < lane && d == my_d) first_of_rank = false;
    }
    if (lane < p.RP) {
        const bool has = lane < p.R && ((own >> lane) & 1u);
        p.send_slot[tok * p.RP + lane] = has ? cnt : -1;
        p.dest_weight[tok * p.RP + lane] = has ? wsum : 0.0f;
    }
    if (lane < K) {
        if (my_e < -1 || my_e >= p.E) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_EXPERT_ID);
        else if (my_d >= 0) atomicAdd(p.counts + my_e, 1);
        if (p.topk_dest != nullptr)  // first slot of each rank carries its message
            p.topk_dest[tok * K + lane] = (int8_t)(first_of_rank ? my_d : -1);
    }
    for (uint32_t b = own; b != 0; b &= b - 1) {  // uniform over the warp
        const int d = __ffs(b) - 1;
        const int slot = __shfl_sync(kFull, cnt, d);
        const size_t row = ((size_t)d * p.R + s) * p.m + slot;
        if (lane == 0) p.src_token[row] = t;
        if (lane < K) {
            const bool local = my_d == d;  // (d is active)
            p.recv_ids[row * K + lane] = local ? my_e : -1;
            p.recv_w[row * K + lane] = local ? my_w : 0.0f;
        }
    }
    if (t == p.T - 1 && lane < p.R)
        p.recv_counts[lane * p.R + s] = cnt + (int)((own >> lane) & 1u);
}

template <int KT>
__global__ void __launch_bounds__(32) dispatch_small_kernel(const DispatchSmallParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x;
    const int K = KT > 0 ? KT : p.K;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * p.stage_bytes);
    if (lane == 0) {
        for (int i = 0; i < kStages; ++i) ptx::mbar_init(&bars[i], 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();

    // Units (< 2^16: at most 32 x 256 tokens x 8 chunks) in 32-bit
    // arithmetic; divisions by chunks and T as multiply-highs.
    const int units = (int)p.units;
    const int first = blockIdx.x, step = gridDim.x;
    const int n = first < units ? (units - 1 - first) / step + 1 : 0;
    auto unit_bytes = [&](int chunk) -> uint32_t {
        const int left = p.row_bytes - chunk * p.chunk_bytes;
        return (uint32_t)(left < p.chunk_bytes ? left : p.chunk_bytes);
    };
    auto issue_x = [&](int i) {  // lane 0: the unit's x chunk into its stage
        const int u = first + i * step;
        const int tok = div_by(u, p.chunks_magic);
        const int chunk = u - tok * p.chunks;
        const int stage = i & (kStages - 1);
        const uint32_t bytes = unit_bytes(chunk);
        ptx::mbar_arrive_expect_tx(&bars[stage], bytes);
        ptx::bulk_g2s(smem + (size_t)stage * p.stage_bytes,
                      p.x + (long long)tok * p.row_bytes + (long long)chunk * p.chunk_bytes,
                      bytes, &bars[stage]);
    };

    // x is an input of the call: request the first chunks right away.
    const int prologue = n < kStages ? n : kStages;
    if (lane == 0)
        for (int i = 0; i < prologue; ++i) issue_x(i);
    int issued = prologue, failed = -1;
    bool ok = true, waited = false;

    for (int i = 0; i < n && ok; ++i) {
        const int u = first + i * step;
        const int tok = div_by(u, p.chunks_magic);   // s * T + t
        const int chunk = u - tok * p.chunks;
        const int s = div_by(tok, p.T_magic), t = tok - s * p.T;
        const int32_t *src_ids = p.topk_ids + (size_t)s * p.T * K;

        // the token's own ids and weights, one per lane (K <= 32)
        const int my_e = lane < K ? __ldg(src_ids + (size_t)t * K + lane) : -1;
        const float my_w = lane < K ? __ldg(p.topk_w + tok * K + lane) : 0.0f;

        // ---- slots: lane d counts the earlier tokens of source s sent to d ----
        int cnt;
        uint32_t own;
        token_slots<KT>(src_ids, t, K, p.E, p.R, p.epr_magic, p.active, lane, cnt, own);

        // The ids are inputs too; before the first write, wait for the kernels
        // before this one in the stream (a combine still reading the
        // previous dispatch's tables).
        if (!waited) {
            ptx::grid_dependency_wait();
            waited = true;
        }

        // ---- routing outputs, by the warp holding the token's first chunk ----
        if (chunk == 0) write_routing(p, K, tok, s, t, my_e, my_w, cnt, own, lane);

        // ---- the row copy: the chunk to every destination row ----
        const int stage = i & (kStages - 1);
        const uint32_t parity = (uint32_t)(i / kStages) & 1u;
        bool ready = true;
        if (lane == 0) ready = ptx::mbar_wait_bounded(&bars[stage], parity, kWaitLimit);
        if (!__shfl_sync(kFull, ready, 0)) {
            ok = false;
            failed = i;
            break;
        }
        const uint8_t *buf = smem + (size_t)stage * p.stage_bytes;
        const uint32_t bytes = unit_bytes(chunk);
        const long long col = (long long)chunk * p.chunk_bytes;
        for (uint32_t b = own; b != 0; b &= b - 1) {
            const int d = __ffs(b) - 1;
            const int slot = __shfl_sync(kFull, cnt, d);
            if (lane == 0)
                ptx::bulk_s2g(p.recv_x + (((long long)d * p.R + s) * p.m + slot) * p.row_bytes +
                                  col,
                              buf, bytes);
        }
        if (lane == 0) {
            ptx::bulk_commit();
            // refill the stage of unit i - 1 once its stores left shared memory
            if (i >= 1 && issued < n) {
                ptx::bulk_wait_read<1>();
                issue_x(issued);
            }
        }
        if (i >= 1 && issued < n) ++issued;
    }
    if (!waited) ptx::grid_dependency_wait();  // (a CTA whose units all failed)
    if (blockIdx.x == 0)  // the next call's counts buffer starts at zero
        for (int e = lane; e < p.E; e += 32) p.counts_clear[e] = 0;

    if (lane == 0) {
        ptx::bulk_wait_all();
        if (!ok) {
            atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
            // chunks requested after the one that timed out, still landing in
            // shared memory, before the CTA exits
            for (int j = failed + 1; j < issued; ++j)
                ptx::mbar_wait_bounded(&bars[j & (kStages - 1)], (uint32_t)(j / kStages) & 1u,
                                       kWaitLimit);
        }
    }
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// FP8 receive rows, one CTA per token: thread 0 requests the bf16 row into
// shared memory, warp 0 derives the token's slots and writes its routing
// outputs (as the bf16 kernel's first-chunk warp), every thread takes VPT
// vectors of the row; the row's amax is one CTA reduction (the same
// barrier publishes the destination rows), and each thread stores the e4m3
// codes of its vectors to every destination row (fp8.cuh's quotient).
template <int KT, int VPT>
__global__ void __launch_bounds__(kSmallFp8MaxThreads)
    dispatch_small_fp8_kernel(const DispatchSmallFp8Params p) {
    extern __shared__ __align__(128) uint8_t row_smem[];  // the token's bf16 row
    __shared__ uint64_t bar;
    __shared__ long long rows[kMaxRanks];                  // destination rows (-1: none)
    __shared__ float red[kSmallFp8MaxThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x, nw = nt >> 5;
    const int K = KT > 0 ? KT : p.K;
    const int tok = blockIdx.x;  // s * T + t, below 2^13
    const int s = div_by(tok, p.T_magic), t = tok - s * p.T;
    const uint32_t row_bytes = (uint32_t)p.H * 2;

    if (tid == 0) {  // x is an input of the call: requested right away
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
        ptx::mbar_arrive_expect_tx(&bar, row_bytes);
        ptx::bulk_g2s(row_smem, p.x + (size_t)tok * p.H, row_bytes, &bar);
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it

    if (warp == 0) {
        const int32_t *src_ids = p.topk_ids + (size_t)s * p.T * K;
        const int my_e = lane < K ? __ldg(src_ids + (size_t)t * K + lane) : -1;
        const float my_w = lane < K ? __ldg(p.topk_w + (size_t)tok * K + lane) : 0.0f;
        int cnt;
        uint32_t own;
        token_slots<KT>(src_ids, t, K, p.E, p.R, p.epr_magic, p.active, lane, cnt, own);
        ptx::grid_dependency_wait();  // before the first write
        write_routing(p, K, tok, s, t, my_e, my_w, cnt, own, lane);
        if (lane < p.RP)
            rows[lane] = (lane < p.R && ((own >> lane) & 1u))
                             ? ((long long)lane * p.R + s) * p.m + cnt
                             : -1;
    } else {
        ptx::grid_dependency_wait();
    }
    if (blockIdx.x == 0)  // the next call's counts buffer starts at zero
        for (int e = tid; e < p.E; e += nt) p.counts_clear[e] = 0;

    const bool landed = ptx::mbar_wait_bounded(&bar, 0, kWaitLimit);
    const uint4 *row = reinterpret_cast<const uint4 *>(row_smem);
    uint4 cur[VPT];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int c = tid + j * nt;
        cur[j] = (landed && c < p.H8) ? row[c] : make_uint4(0, 0, 0, 0);
        const uint32_t u[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(lo_f(u[e])), fabsf(hi_f(u[e]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    if (lane == 0) red[warp] = amax;
    if (!__syncthreads_and(landed)) {  // (also publishes rows[] and red[])
        if (tid == 0) {
            atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
            // the row copy lands before the shared memory goes away
            ptx::mbar_wait_bounded(&bar, 0, kWaitLimit);
        }
        return;
    }
    amax = red[0];
    for (int w = 1; w < nw; ++w) amax = fmaxf(amax, red[w]);
    const fp8::RowScale rs = fp8::row_scale(amax);
    float f[VPT][8];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const uint32_t u[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[j][2 * e] = lo_f(u[e]);
            f[j][2 * e + 1] = hi_f(u[e]);
        }
    }
    uint2 q[VPT];
    fp8::quantize_row<VPT>(f, rs, q);
    for (int d = 0; d < p.RP; ++d) {
        const long long dst_row = rows[d];
        if (dst_row < 0) continue;
        uint2 *dst = reinterpret_cast<uint2 *>(p.recv_x8 + dst_row * p.H);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = tid + j * nt;
            if (c < p.H8) __stcs(dst + c, q[j]);
        }
        if (tid == 0) p.recv_scale[dst_row] = rs.s;
    }
}

}  // namespace

cudaError_t dispatch_small_prepare(int row_bytes, int num_sms, DispatchSmallShapes *out) {
    // For 1..8 chunks per row: chunk bytes (a multiple of 16, bulk copies),
    // two stages of shared memory, CTAs per SM from the occupancy (at most 16).
    const int max_stage = (row_bytes + 15) / 16 * 16;
    const size_t max_smem = 2 * (size_t)((max_stage + 127) / 128 * 128) + 2 * sizeof(uint64_t);
    const void *kern[5] = {(const void *)dispatch_small_kernel<0>,
                           (const void *)dispatch_small_kernel<1>,
                           (const void *)dispatch_small_kernel<2>,
                           (const void *)dispatch_small_kernel<4>,
                           (const void *)dispatch_small_kernel<8>};
    for (const void *k : kern) {
        cudaError_t err = raise_smem_limit(k, max_smem);
        if (err != cudaSuccess) return err;
    }
    out->stages = kStages;
    for (int c = 1; c <= kSmallMaxChunks; ++c) {
        int chunk = (row_bytes + c - 1) / c;
        chunk = (chunk + 15) / 16 * 16;
        const int stage_bytes = (chunk + 127) / 128 * 128;
        const size_t smem = (size_t)out->stages * stage_bytes + out->stages * sizeof(uint64_t);
        int per_sm = 0;
        cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, dispatch_small_kernel<8>, 32, smem);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        if (per_sm > 16) per_sm = 16;
        out->chunk_bytes[c] = chunk;
        out->chunks[c] = (row_bytes + chunk - 1) / chunk;
        out->stage_bytes[c] = stage_bytes;
        out->shape[c].grid = num_sms * per_sm;
        out->shape[c].block = 32;
        out->shape[c].smem = smem;
    }
    return cudaSuccess;
}

int dispatch_small_chunks(int row_bytes, int num_sms, long long tokens) {
    // about four units per SM, 1..8 chunks per row, chunks of at least 1 KB
    const long long t = tokens > 0 ? tokens : 1;
    long long c = (4LL * num_sms + t - 1) / t;
    c = c < 1 ? 1 : (c > kSmallMaxChunks ? kSmallMaxChunks : c);
    while (c > 1 && row_bytes / c < 1024) --c;
    return (int)c;
}

cudaError_t launch_dispatch_small(const DispatchSmallParams &pc, const LaunchShape &shape,
                                  cudaStream_t st) {
    DispatchSmallParams p = pc;
    p.epr_magic = owner_magic(p.Epr);
    if (p.T < 1 || p.T > kRouteTile || p.R > kMaxRanks || p.K > kMaxTopK ||
        p.stages != kStages || p.chunks < 1 || p.chunks > kSmallMaxChunks ||
        p.units != (long long)p.R * p.T * p.chunks)
        return cudaErrorInvalidValue;
    p.chunks_magic = div_magic(p.chunks);  // exact: units < 2^16, chunks <= 8
    p.T_magic = div_magic(p.T);            // exact: tokens < 2^13, T <= 256
    long long grid = shape.grid;
    if (grid > p.units) grid = p.units;
    if (grid < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = shape.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (p.K) {
        case 1: return cudaLaunchKernelEx(&cfg, dispatch_small_kernel<1>, p);
        case 2: return cudaLaunchKernelEx(&cfg, dispatch_small_kernel<2>, p);
        case 4: return cudaLaunchKernelEx(&cfg, dispatch_small_kernel<4>, p);
        case 8: return cudaLaunchKernelEx(&cfg, dispatch_small_kernel<8>, p);
        default: return cudaLaunchKernelEx(&cfg, dispatch_small_kernel<0>, p);
    }
}


namespace {

// Threads for a row of H8 16-byte vectors: 128 while the row fits in 8
// vectors per thread, else the fewest whole warps that cover it with 8.
int fp8_threads(int H8) {
    if (H8 <= 8 * 128) return 128;
    return ((H8 + 7) / 8 + 31) / 32 * 32;
}

template <int VPT>
struct SmallFp8 {
    static cudaError_t attr(size_t smem) {
        cudaError_t e = raise_smem_limit(dispatch_small_fp8_kernel<8, VPT>, smem);
        if (e != cudaSuccess) return e;
        return raise_smem_limit(dispatch_small_fp8_kernel<0, VPT>, smem);
    }
    static cudaError_t launch(const DispatchSmallFp8Params &p, const DispatchSmallFp8Shape &sh,
                              cudaStream_t st) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(p.R * p.T), 1, 1);
        cfg.blockDim = dim3((unsigned)sh.threads, 1, 1);
        cfg.dynamicSmemBytes = sh.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (p.K == 8) return cudaLaunchKernelEx(&cfg, dispatch_small_fp8_kernel<8, VPT>, p);
        return cudaLaunchKernelEx(&cfg, dispatch_small_fp8_kernel<0, VPT>, p);
    }
};

template <template <int> class F, typename Fn>
cudaError_t by_vpt(int vpt, Fn fn) {
    switch (vpt) {
        case 1: return fn(F<1>());
        case 2: return fn(F<2>());
        case 3: return fn(F<3>());
        case 4: return fn(F<4>());
        case 5: return fn(F<5>());
        case 6: return fn(F<6>());
        case 7: return fn(F<7>());
        case 8: return fn(F<8>());
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t dispatch_small_fp8_prepare(int H, DispatchSmallFp8Shape *out) {
    if (H % 16 != 0 || H / 8 > 2048) return cudaErrorInvalidValue;
    const int H8 = H / 8;
    out->threads = fp8_threads(H8);
    out->vpt = (H8 + out->threads - 1) / out->threads;
    out->smem = (size_t)H * 2;
    if (out->threads > kSmallFp8MaxThreads) return cudaErrorInvalidValue;
    const size_t smem = out->smem;
    return by_vpt<SmallFp8>(out->vpt, [&](auto f) { return decltype(f)::attr(smem); });
}

cudaError_t launch_dispatch_small_fp8(const DispatchSmallFp8Params &pc,
                                      const DispatchSmallFp8Shape &shape, cudaStream_t st) {
    DispatchSmallFp8Params p = pc;
    if (p.T < 1 || p.T > kRouteTile || p.R > kMaxRanks || p.K > kMaxTopK || p.H % 16 != 0 ||
        p.H8 != p.H / 8 || shape.smem != (size_t)p.H * 2 ||
        (long long)shape.threads * shape.vpt < p.H8)
        return cudaErrorInvalidValue;
    p.epr_magic = owner_magic(p.Epr);
    p.T_magic = div_magic(p.T);  // exact: tokens < 2^13, T <= 256
    return by_vpt<SmallFp8>(shape.vpt, [&](auto f) { return decltype(f)::launch(p, shape, st); });
}

}  // namespace moe
