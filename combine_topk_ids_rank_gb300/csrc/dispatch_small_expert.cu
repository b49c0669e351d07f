// dispatch_small_expert.cu -- the expert-major layout's dispatch phase in one
// launch, for small batches.
//
// Operation: the same as route_expert.cu + the row copy (InferenceX PR
// #2450, "CollectiveX: add FlashInfer one-sided NVLink EP for the GB SKUs":
// the low-latency padded layouts, whose received rows carry one expert
// each).  Readings as in route_expert.cu: expert e has a plane of cap = R * m
// rows; one row per distinct (token, expert) with a valid id on an active
// rank, in ascending (source rank, token):
//   row(s,t,e) = e * cap + #{(s',t') before (s,t) whose ids include e},
//   recv_x[row][:] = x[s][t][:],
// with send_row / wsum per top-k slot, src_token and recv_w per row, the
// rows per expert (recv_counts) and the expert histogram (duplicates
// included) of the routing passes.
//
// GB300 design, for batches where launches and dependent round trips cost
// more than the bytes: one-warp CTAs, several per SM, each taking units (a
// token row, or a chunk of it when there are few tokens) of the grid-strided
// unit list, as the rank layout's one-launch dispatch does.  Lane k holds the
// token's k-th expert; the token's rows come from the ids of every token
// before it in (source, token) order, one warp ballot per top-k slot and 32
// earlier tokens, so no CTA waits for another.  Meanwhile lane 0 has
// requested the unit's x chunk into a shared-memory stage with a bulk copy;
// once the rows are known it stores the chunk to each of them with bulk
// shared -> global copies.  The warp holding a token's first chunk writes its
// send row, weights, source-map entries and row weights, and adds to the two
// count arrays with atomics.  Both count arrays live in one of two buffer
// pairs that alternate between calls: each call adds into the pair the
// previous call cleared and clears the other one.  Waits are bounded: on
// time-out the kernel raises the flag, drains its copies and returns.
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

// Expert id if it is valid and lives on an active rank, else -1.
__device__ __forceinline__ int live_expert(int e, int E, unsigned long long epr_magic,
                                           uint32_t active) {
    if (e < 0 || e >= E) return -1;
    return ((active >> owner_of(e, epr_magic)) & 1u) ? e : -1;
}

// Lane k: how many tokens before `tok` (flat index s * T + t) carry my_e,
// the lane's own live expert (lanes without one count nothing).  One ballot
// per top-k slot and 32 earlier tokens; a token carrying an expert twice
// counts once.  The ids of G groups of 32 tokens are loaded together (G * K
// registers, at most 32), so the scan waits for one round trip per G groups.
template <int KT>
__device__ __forceinline__ int rows_before(const int32_t *ids_all, int tok, int K, int my_e,
                                           int lane) {
    constexpr int KA = KT > 0 ? KT : kMaxTopK;
    constexpr int G = KA >= 32 ? 1 : (32 / KA > 8 ? 8 : 32 / KA);
    int ek[KA];
#pragma unroll
    for (int k = 0; k < KA; ++k) ek[k] = __shfl_sync(kFull, my_e, k & 31);
    int cnt = 0;
    for (int base = 0; base < tok; base += 32 * G) {
        int ids[G][KA];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int tt = base + 32 * g + lane;
#pragma unroll
            for (int k = 0; k < KA; ++k)
                ids[g][k] = (tt < tok && k < K) ? __ldg(ids_all + (size_t)tt * K + k) : -1;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (base + 32 * g >= tok) break;  // (uniform over the warp)
#pragma unroll
            for (int k = 0; k < KA; ++k) {
                if (k >= K) break;
                bool has = false;
#pragma unroll
                for (int k2 = 0; k2 < KA; ++k2)
                    if (k2 < K) has |= ids[g][k2] == ek[k];
                const uint32_t b = __ballot_sync(kFull, has && ek[k] >= 0);
                if (lane == k) cnt += __popc(b);
            }
        }
    }
    return cnt;
}

// The routing outputs of token `tok` (one warp; its raw ids, live experts
// and weights one per lane, first_of_e and my_row per lane as the kernels
// derive them): send row and weights of every top-k slot (padding slots up
// to KP included), source map and row weight of each of its rows, the two
// count arrays, the bad-id flag.
template <class P>
__device__ __forceinline__ void write_expert_routing(const P &p, int K, int tok, int raw,
                                                     int my_e, float my_w, bool first_of_e,
                                                     long long my_row, int lane) {
    // slot k's weight: its expert's weights over k' >= k in ascending k',
    // from +0.0 (only the first slot of an expert keeps it)
    float wsum = 0.0f;
    for (int k = 0; k < K; ++k) {
        const int e = __shfl_sync(kFull, my_e, k);
        const float wk = __shfl_sync(kFull, my_w, k);
        if (k >= lane && e == my_e && my_e >= 0) wsum = __fadd_rn(wsum, wk);
    }
    const long long trow = (long long)tok * p.KP;
    if (lane < K) {
        p.send_row[trow + lane] = (int32_t)my_row;
        p.wsum[trow + lane] = first_of_e ? wsum : 0.0f;
        if (raw < -1 || raw >= p.E) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_EXPERT_ID);
        if (my_e >= 0) atomicAdd(p.counts + my_e, 1);
        if (first_of_e) {
            p.src_token[my_row] = tok;  // s * T + t (uniform T)
            p.recv_w[my_row] = wsum;
            atomicAdd(p.recv_counts + my_e, 1);
        }
    } else if (lane < p.KP) {
        p.send_row[trow + lane] = -1;
        p.wsum[trow + lane] = 0.0f;
    }
}

// Lane k's live expert of token `tok`, whether slot k is its first, and its
// row (-1 if none); raw id and weight of slot k.
template <int KT, class P>
__device__ __forceinline__ void token_rows(const P &p, int K, int tok, int lane, int &raw,
                                           int &my_e, float &my_w, bool &first_of_e,
                                           long long &my_row) {
    raw = lane < K ? __ldg(p.topk_ids + (size_t)tok * K + lane) : -1;
    my_w = lane < K ? __ldg(p.topk_w + (size_t)tok * K + lane) : 0.0f;
    my_e = live_expert(raw, p.E, p.epr_magic, p.active);
    first_of_e = my_e >= 0;
    for (int k = 0; k < K; ++k) {
        const int e = __shfl_sync(kFull, my_e, k);
        if (k < lane && e == my_e) first_of_e = false;
    }
    const int before = rows_before<KT>(p.topk_ids, tok, K, my_e, lane);
    my_row = first_of_e ? (long long)my_e * p.cap + before : -1;  // before < R*T <= cap
}

template <int KT>
__global__ void __launch_bounds__(32)
    dispatch_small_expert_kernel(const DispatchSmallExpertParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x;
    const int K = KT > 0 ? KT : p.K;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * p.stage_bytes);
    if (lane == 0) {
        for (int i = 0; i < kStages; ++i) ptx::mbar_init(&bars[i], 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();

    // Units (at most 32 x 256 tokens x 8 chunks) in 32-bit arithmetic; the
    // division by chunks as a multiply-high (tokens are flat: s * T + t).
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
        const int tok = div_by(u, p.chunks_magic);  // s * T + t
        const int chunk = u - tok * p.chunks;

        // the token's ids and weights, one per lane (K <= 32), and its rows
        int raw, my_e;
        float my_w;
        bool first_of_e;
        long long my_row;
        token_rows<KT>(p, K, tok, lane, raw, my_e, my_w, first_of_e, my_row);

        // The ids are inputs too; before the first write, wait for the kernels
        // before this one in the stream (a combine still reading the
        // previous dispatch's tables).
        if (!waited) {
            ptx::grid_dependency_wait();
            waited = true;
        }

        // ---- routing outputs, by the warp holding the token's first chunk ----
        if (chunk == 0) write_expert_routing(p, K, tok, raw, my_e, my_w, first_of_e, my_row, lane);

        // ---- the row copy: the chunk to every row of the token ----
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
        for (int k = 0; k < K; ++k) {  // uniform over the warp
            const long long row = __shfl_sync(kFull, my_row, k);
            if (row >= 0 && lane == 0)
                ptx::bulk_s2g(p.recv_x + row * p.row_bytes + col, buf, bytes);
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
    if (blockIdx.x == 0)  // the next call's count buffers start at zero
        for (int e = lane; e < p.E; e += 32) {
            p.counts_clear[e] = 0;
            p.recv_counts_clear[e] = 0;
        }

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

constexpr int kFp8MaxThreads = 256;  // threads of the FP8 kernel: at most

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// FP8 receive rows, one CTA per token: thread 0 requests the bf16 row into
// shared memory, warp 0 finds the token's rows and writes its routing
// outputs (as the bf16 kernel's first-chunk warp), every thread takes VPT
// vectors of the row; the row's amax is one CTA reduction (the same
// barrier publishes the rows), and each thread stores the e4m3 codes of its
// vectors to every row of the token (fp8.cuh's quotient).
template <int KT, int VPT>
__global__ void __launch_bounds__(kFp8MaxThreads)
    dispatch_small_expert_fp8_kernel(const DispatchSmallExpertFp8Params p) {
    extern __shared__ __align__(128) uint8_t row_smem[];  // the token's bf16 row
    __shared__ uint64_t bar;
    __shared__ long long rows[kMaxTopK];                   // by top-k slot (-1: none)
    __shared__ float red[kFp8MaxThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x, nw = nt >> 5;
    const int K = KT > 0 ? KT : p.K;
    const int tok = blockIdx.x;  // s * T + t, below 2^13
    const uint32_t row_bytes = (uint32_t)p.H * 2;

    if (tid == 0) {  // x is an input of the call: requested right away
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
        ptx::mbar_arrive_expect_tx(&bar, row_bytes);
        ptx::bulk_g2s(row_smem, p.x + (size_t)tok * p.H, row_bytes, &bar);
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it

    if (warp == 0) {
        int raw, my_e;
        float my_w;
        bool first_of_e;
        long long my_row;
        token_rows<KT>(p, K, tok, lane, raw, my_e, my_w, first_of_e, my_row);
        ptx::grid_dependency_wait();  // before the first write
        write_expert_routing(p, K, tok, raw, my_e, my_w, first_of_e, my_row, lane);
        if (lane < K) rows[lane] = my_row;
    } else {
        ptx::grid_dependency_wait();
    }
    if (blockIdx.x == 0)  // the next call's count buffers start at zero
        for (int e = tid; e < p.E; e += nt) {
            p.counts_clear[e] = 0;
            p.recv_counts_clear[e] = 0;
        }

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
    for (int k = 0; k < K; ++k) {
        const long long dst_row = rows[k];
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

// Threads for a row of H8 16-byte vectors: 128 while the row fits in 8
// vectors per thread, else the fewest whole warps that cover it with 8.
int fp8_threads(int H8) {
    if (H8 <= 8 * 128) return 128;
    return ((H8 + 7) / 8 + 31) / 32 * 32;
}

template <int VPT>
struct ExpertFp8 {
    static cudaError_t attr(size_t smem) {
        cudaError_t e = raise_smem_limit(dispatch_small_expert_fp8_kernel<8, VPT>, smem);
        if (e != cudaSuccess) return e;
        return raise_smem_limit(dispatch_small_expert_fp8_kernel<0, VPT>, smem);
    }
    static cudaError_t launch(const DispatchSmallExpertFp8Params &p,
                              const DispatchSmallFp8Shape &sh, cudaStream_t st) {
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
        if (p.K == 8) return cudaLaunchKernelEx(&cfg, dispatch_small_expert_fp8_kernel<8, VPT>, p);
        return cudaLaunchKernelEx(&cfg, dispatch_small_expert_fp8_kernel<0, VPT>, p);
    }
};

template <typename Fn>
cudaError_t by_vpt(int vpt, Fn fn) {
    switch (vpt) {
        case 1: return fn(ExpertFp8<1>());
        case 2: return fn(ExpertFp8<2>());
        case 3: return fn(ExpertFp8<3>());
        case 4: return fn(ExpertFp8<4>());
        case 5: return fn(ExpertFp8<5>());
        case 6: return fn(ExpertFp8<6>());
        case 7: return fn(ExpertFp8<7>());
        case 8: return fn(ExpertFp8<8>());
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t dispatch_small_expert_fp8_prepare(int H, DispatchSmallFp8Shape *out) {
    if (H % 16 != 0 || H / 8 > 2048) return cudaErrorInvalidValue;
    const int H8 = H / 8;
    out->threads = fp8_threads(H8);
    out->vpt = (H8 + out->threads - 1) / out->threads;
    out->smem = (size_t)H * 2;
    if (out->threads > kFp8MaxThreads) return cudaErrorInvalidValue;
    const size_t smem = out->smem;
    return by_vpt(out->vpt, [&](auto f) { return decltype(f)::attr(smem); });
}

cudaError_t launch_dispatch_small_expert_fp8(const DispatchSmallExpertFp8Params &pc,
                                             const DispatchSmallFp8Shape &shape,
                                             cudaStream_t st) {
    DispatchSmallExpertFp8Params p = pc;
    if (p.T < 1 || p.T > kRouteTile || p.R < 1 || p.R > kMaxRanks || p.K < 1 ||
        p.K > kMaxTopK || p.KP < p.K || p.KP > 32 || p.E < p.R || p.E % p.R != 0 ||
        p.Epr != p.E / p.R || p.cap < p.R * p.T || p.H % 16 != 0 || p.H8 != p.H / 8 ||
        shape.smem != (size_t)p.H * 2 || shape.threads > kFp8MaxThreads ||
        (long long)shape.threads * shape.vpt < p.H8)
        return cudaErrorInvalidValue;
    p.epr_magic = owner_magic(p.Epr);  // exact: e < E <= 1024 experts
    return by_vpt(shape.vpt, [&](auto f) { return decltype(f)::launch(p, shape, st); });
}

cudaError_t dispatch_small_expert_prepare(int row_bytes, int num_sms, DispatchSmallShapes *out) {
    // For 1..8 chunks per row: chunk bytes (a multiple of 16, bulk copies),
    // two stages of shared memory, CTAs per SM from the occupancy (at most 16).
    const int max_stage = (row_bytes + 15) / 16 * 16;
    const size_t max_smem = 2 * (size_t)((max_stage + 127) / 128 * 128) + 2 * sizeof(uint64_t);
    const void *kern[5] = {(const void *)dispatch_small_expert_kernel<0>,
                           (const void *)dispatch_small_expert_kernel<1>,
                           (const void *)dispatch_small_expert_kernel<2>,
                           (const void *)dispatch_small_expert_kernel<4>,
                           (const void *)dispatch_small_expert_kernel<8>};
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
            &per_sm, dispatch_small_expert_kernel<8>, 32, smem);
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

cudaError_t launch_dispatch_small_expert(const DispatchSmallExpertParams &pc,
                                         const LaunchShape &shape, cudaStream_t st) {
    DispatchSmallExpertParams p = pc;
    if (p.T < 1 || p.T > kRouteTile || p.R < 1 || p.R > kMaxRanks || p.K < 1 ||
        p.K > kMaxTopK || p.KP < p.K || p.KP > 32 || p.E < p.R || p.E % p.R != 0 ||
        p.Epr != p.E / p.R || p.cap < p.R * p.T || p.stages != kStages || p.chunks < 1 ||
        p.chunks > kSmallMaxChunks || p.units != (long long)p.R * p.T * p.chunks ||
        p.chunk_bytes * p.chunks < p.row_bytes || p.chunk_bytes > p.stage_bytes)
        return cudaErrorInvalidValue;
    p.epr_magic = owner_magic(p.Epr);      // exact: e < E <= 1024 experts
    p.chunks_magic = div_magic(p.chunks);  // exact: units < 2^17, chunks <= 8
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
        case 1: return cudaLaunchKernelEx(&cfg, dispatch_small_expert_kernel<1>, p);
        case 2: return cudaLaunchKernelEx(&cfg, dispatch_small_expert_kernel<2>, p);
        case 4: return cudaLaunchKernelEx(&cfg, dispatch_small_expert_kernel<4>, p);
        case 8: return cudaLaunchKernelEx(&cfg, dispatch_small_expert_kernel<8>, p);
        default: return cudaLaunchKernelEx(&cfg, dispatch_small_expert_kernel<0>, p);
    }
}

}  // namespace moe
