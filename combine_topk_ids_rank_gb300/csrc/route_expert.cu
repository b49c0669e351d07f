// route_expert.cu -- routing for the expert-major receive layout, where
// every received row carries a single expert.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs": the association-order analysis -- backends
// whose received rows carry one expert each, the low-latency padded
// layouts; the harness review -- those backends apply the gates in the
// combine kernel, "weighted-kernel-sum").  Readings:
//   expert e has a plane of cap = R * m rows; one row per distinct
//   (token, expert) with a valid id on an active rank, in ascending
//   (source rank, token);
//   send_row[s][t][k] = e_k * cap + slot for the first k carrying that
//   expert, -1 for later duplicates, absent ids and padding entries k >= K;
//   wsum[s][t][k] = sum over the token's k' >= k with the same expert, in
//   ascending k', of w[k'] from +0.0f (0 where send_row is -1);
//   recv_counts[e], src_token[e][slot] = s * stride + t, recv_w[e][slot].
//
// Two passes over tiles of 256 tokens of one source rank (one token per
// thread), grid = tiles x R:
//   pass 1 (route_e_count): each warp marks, per expert, the lanes whose
//          token carries it (shared-memory lane masks, atomicOr), then the
//          tile's rows per expert are the popcounts, written to
//          tile_counts[s][tile][e]; the expert histogram (duplicates
//          included) into an accumulator that pass 2 moves to
//          local_expert_counts and clears; the bad-id flag.
//   pass 2 (route_e_scan): rebuilds the masks while pass 1 still runs
//          (programmatic dependent launch), sums the counts of every
//          earlier (source, tile) per expert -- O(tiles * E) reads per CTA,
//          split over the CTA's threads in interleaved partial sums when
//          there are fewer experts than threads -- and gives
//          each (token, expert) its row: that base + the popcounts of the
//          earlier warps' masks + the popcount of its own warp's mask
//          below its lane.  Grid z splits the top-k slots into groups of
//          kg (all KP, or one slot per CTA when the batch is small); every
//          CTA rebuilds the masks and bases it needs.  The last CTA writes
//          recv_counts.
#include "kernels.h"
#include "ptx.cuh"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr int kTile = 256;
constexpr int kWarps = kTile / 32;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Expert id of slot k if it is valid and lives on an active rank, else -1.
__device__ __forceinline__ int live_expert(int e, const RouteExpertParams &p) {
    if (e < 0 || e >= p.E) return -1;
    return ((p.active >> (e / p.Epr)) & 1u) ? e : -1;
}

template <int KT>
__device__ __forceinline__ void load_ids(const RouteExpertParams &p, int s, int t, int K,
                                         int (&ids)[KT > 0 ? KT : kMaxTopK]) {
    const int32_t *src = p.topk_ids + ((size_t)s * p.map.stride + t) * K;
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : kMaxTopK); ++k) ids[k] = k < K ? src[k] : -1;
}

template <int KT>
__global__ void __launch_bounds__(kTile) route_e_count_kernel(const RouteExpertParams p) {
    constexpr int KA = KT > 0 ? KT : kMaxTopK;
    __shared__ uint32_t masks[kWarps][kMaxExpertsExpertLayout];
    __shared__ int32_t hist[kMaxExpertsExpertLayout];
    const int tile = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = tile * kTile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;

    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    for (int i = threadIdx.x; i < kWarps * p.E; i += kTile) masks[i / p.E][i % p.E] = 0u;
    for (int e = threadIdx.x; e < p.E; e += kTile) hist[e] = 0;
    __syncthreads();

    if (t < p.map.count[s]) {
        int ids[KA];
        load_ids<KT>(p, s, t, K, ids);
        bool bad = false;
#pragma unroll
        for (int k = 0; k < KA; ++k) {
            const int e = ids[k];
            if (e == -1) continue;
            if (e < -1 || e >= p.E) {
                bad = true;
                continue;
            }
            if (live_expert(e, p) < 0) continue;
            atomicAdd(&hist[e], 1);
            atomicOr(&masks[warp][e], 1u << lane);
        }
        if (bad) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_EXPERT_ID);
    }
    __syncthreads();

    int32_t *counts = p.tile_counts + ((size_t)s * p.ntiles + tile) * p.E;
    for (int e = threadIdx.x; e < p.E; e += kTile) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c += __popc(masks[w][e]);
        counts[e] = c;
        if (hist[e] != 0) atomicAdd(&p.hist_accum[e], hist[e]);
    }
}

template <int KT>
__global__ void __launch_bounds__(kTile) route_e_scan_kernel(const RouteExpertParams p) {
    constexpr int KA = KT > 0 ? KT : kMaxTopK;
    __shared__ uint32_t masks[kWarps][kMaxExpertsExpertLayout];
    __shared__ int32_t base[kMaxExpertsExpertLayout];
    __shared__ int32_t part_sum[kTile > kMaxExpertsExpertLayout ? kTile : kMaxExpertsExpertLayout];
    const int tile = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = tile * kTile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;
    const bool has_token = t < p.map.count[s];
    const int k_lo = (int)blockIdx.z * p.kg, k_hi = k_lo + p.kg;  // this CTA's slots
    ptx::launch_dependents();  // the row copy may start loading its inputs

    // Inputs of the call: loaded and marked before the count pass finishes.
    for (int i = threadIdx.x; i < kWarps * p.E; i += kTile) masks[i / p.E][i % p.E] = 0u;
    __syncthreads();
    int ids[KA];
    float w[KA];
    if (has_token) {
        load_ids<KT>(p, s, t, K, ids);
        const float *src = p.topk_w + ((size_t)s * p.map.stride + t) * K;
#pragma unroll
        for (int k = 0; k < KA; ++k) {
            w[k] = k < K ? src[k] : 0.0f;
            ids[k] = live_expert(ids[k], p);
            if (ids[k] >= 0) atomicOr(&masks[warp][ids[k]], 1u << lane);
        }
    }
    ptx::grid_dependency_wait();  // tile counts and histogram of the count pass

    // This CTA's share of the experts: move the histogram out, leave zero.
    {
        const int ncta = p.R * p.ntiles * (int)gridDim.z;
        const int cta = (s * p.ntiles + tile) * (int)gridDim.z + (int)blockIdx.z;
        for (int e = cta + (int)threadIdx.x * ncta; e < p.E; e += kTile * ncta) {
            p.local_counts[e] = __ldcg(p.hist_accum + e);
            p.hist_accum[e] = 0;
        }
    }

    // Rows of this expert that come before this tile: all tiles of earlier
    // sources and the earlier tiles of this source.  With few experts the
    // threads split each expert's (source, tile) range into `parts`
    // interleaved partial sums, so no thread walks a long chain of loads.
    const int before = s * p.ntiles + tile;
    const int parts = p.E >= kTile ? 1 : kTile / p.E;
    for (int x = threadIdx.x; x < p.E * parts; x += kTile) {
        const int e = x % p.E, part = x / p.E;
        int b = 0;
#pragma unroll 4
        for (int i = part; i < before; i += parts) b += p.tile_counts[(size_t)i * p.E + e];
        part_sum[x] = b;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += kTile) {
        int b = 0;
        for (int part = 0; part < parts; ++part) b += part_sum[part * p.E + e];
        base[e] = b;
    }
    __syncthreads();

    if (has_token) {
        const long long tok = (long long)s * p.map.stride + t;
        int32_t *srow = p.send_row + tok * p.KP;
        float *wrow = p.wsum + tok * p.KP;
        const uint32_t lt = lanemask_lt();
#pragma unroll
        for (int k = 0; k < KA; ++k) {
            if (k < k_lo || k >= k_hi) continue;
            const int e = ids[k];
            bool first = e >= 0;
#pragma unroll
            for (int k2 = 0; k2 < k; ++k2)
                if (ids[k2] == e) first = false;
            int32_t row = -1;
            float sum = 0.0f;
            if (first) {
#pragma unroll
                for (int k2 = k; k2 < KA; ++k2)
                    if (ids[k2] == e) sum = __fadd_rn(sum, w[k2]);
                int j = base[e] + __popc(masks[warp][e] & lt);
                for (int w2 = 0; w2 < warp; ++w2) j += __popc(masks[w2][e]);
                row = (int32_t)((long long)e * p.cap + j);
                p.src_token[row] = (int32_t)tok;
                p.recv_w[row] = sum;
            }
            if (k < K) {
                srow[k] = row;
                wrow[k] = sum;
            }
        }
        for (int k = max(K, k_lo); k < min(p.KP, k_hi); ++k) {
            srow[k] = -1;
            wrow[k] = 0.0f;
        }
    }

    if (s == p.R - 1 && tile == p.ntiles - 1 && blockIdx.z == 0) {
        for (int e = threadIdx.x; e < p.E; e += kTile) {
            int c = base[e];
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) c += __popc(masks[w2][e]);
            p.recv_counts[e] = c;
        }
    }
}

template <typename Kern>
cudaError_t launch2d(Kern kern, const RouteExpertParams &p, cudaStream_t st, bool pdl,
                     unsigned gz = 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ntiles, p.R, gz);
    cfg.blockDim = dim3(kTile, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int route_expert_tile() { return kTile; }

cudaError_t launch_route_expert(const RouteExpertParams &p, cudaStream_t st) {
    if (p.E > kMaxExpertsExpertLayout || p.K > kMaxTopK || p.KP < p.K || p.ntiles < 1)
        return cudaErrorInvalidValue;
    // Common top-k values get their own instantiation: the per-slot loops
    // (duplicate checks, weight sums) are unrolled over KT slots, where the
    // generic one runs them over kMaxTopK.
    cudaError_t e;
    switch (p.K) {
        case 1: e = launch2d(route_e_count_kernel<1>, p, st, false); break;
        case 2: e = launch2d(route_e_count_kernel<2>, p, st, false); break;
        case 4: e = launch2d(route_e_count_kernel<4>, p, st, false); break;
        case 8: e = launch2d(route_e_count_kernel<8>, p, st, false); break;
        default: e = launch2d(route_e_count_kernel<0>, p, st, false); break;
    }
    if (e != cudaSuccess) return e;
    if (p.kg < 1 || p.KP % p.kg != 0) return cudaErrorInvalidValue;
    const unsigned gz = (unsigned)(p.KP / p.kg);
    switch (p.K) {
        case 1: return launch2d(route_e_scan_kernel<1>, p, st, true, gz);
        case 2: return launch2d(route_e_scan_kernel<2>, p, st, true, gz);
        case 4: return launch2d(route_e_scan_kernel<4>, p, st, true, gz);
        case 8: return launch2d(route_e_scan_kernel<8>, p, st, true, gz);
        default: return launch2d(route_e_scan_kernel<0>, p, st, true, gz);
    }
}

}  // namespace moe
