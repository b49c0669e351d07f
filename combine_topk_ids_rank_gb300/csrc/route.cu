// route.cu -- routing of top-k expert ids onto logical destination ranks.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs": "Synthesis" table -- duplicate experts on one
// rank are read once, partial routing compacts each plane; "Best remaining
// lead" -- recv counters are the authoritative per-source counts; bring-up
// run table -- expert ids and weights travel as payloads, non-local ids are
// masked, local_expert_counts):
//   dmask(s,t)       = set of ranks owner(e_k) = e_k / Epr over valid k
//   slot(s,t,d)      = #{t' < t : d in dmask(s,t')}   (ascending token order)
//   dest_weight(s,t,d) = sum over k with owner(e_k) = d, ascending k, of w_k
//   recv_counts[d][s], src_token[d][s][slot], masked metadata rows,
//   local_expert_counts[e] = #valid (s,t,k) entries with e_k = e.
//
// Two passes over tiles of 256 tokens of one source rank (grid: tiles x R):
//   pass 1 (route_count): destination mask per token, destination counts
//          and an expert histogram per tile;
//   pass 2 (route_scan):  exclusive prefix of the earlier tiles' counts plus
//          a warp-ballot / cross-warp scan inside the tile gives each
//          token's slot on every destination; then all routing outputs are
//          written, and the per-tile histograms are reduced.
// Both passes are O(T) in work; pass 2 starts early through programmatic
// dependent launch and waits for pass 1 on the device.
#include "kernels.h"
#include "ptx.cuh"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kRouteTile / 32;

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// KT > 0: top_k known at compile time (ids/weights held in registers);
// KT == 0: any top_k, read from global memory (L1) when needed.
template <int KT>
__global__ void __launch_bounds__(kRouteTile)
    route_count_kernel(const RouteCountParams p) {
    extern __shared__ int32_t hist[];  // [E]
    __shared__ int32_t warp_cnt[kWarps][32];
    const int tile = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = tile * kRouteTile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;

    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    for (int e = threadIdx.x; e < p.E; e += kRouteTile) hist[e] = 0;
    __syncthreads();

    uint32_t mask = 0;
    bool bad = false;
    if (t < p.T) {
        const int32_t *ids = p.topk_ids + ((size_t)s * p.T + t) * K;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int e = ids[k];
            if (e == -1) continue;
            if (e < -1 || e >= p.E) {
                bad = true;
                continue;
            }
            mask |= 1u << (e / p.Epr);
            atomicAdd(&hist[e], 1);
        }
        p.dmask[(size_t)s * p.T + t] = mask;
    }
    if (bad) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_EXPERT_ID);

    for (int d = 0; d < p.R; ++d) {
        const uint32_t b = __ballot_sync(kFull, (mask >> d) & 1u);
        if (lane == 0) warp_cnt[warp][d] = __popc(b);
    }
    __syncthreads();

    if (threadIdx.x < p.RP) {
        const int d = threadIdx.x;
        int sum = 0;
        if (d < p.R)
            for (int w = 0; w < kWarps; ++w) sum += warp_cnt[w][d];
        p.tile_counts[((size_t)s * p.ntiles + tile) * p.RP + d] = sum;
    }
    int32_t *th = p.tile_hist + ((size_t)s * p.ntiles + tile) * p.E;
    for (int e = threadIdx.x; e < p.E; e += kRouteTile) th[e] = hist[e];
}

template <int KT>
__global__ void __launch_bounds__(kRouteTile)
    route_scan_kernel(const RouteScanParams p) {
    __shared__ int32_t prefix[32];
    __shared__ int32_t warp_cnt[kWarps][32];
    __shared__ int32_t warp_off[kWarps][32];
    __shared__ int32_t tile_total[32];
    const int tile = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = tile * kRouteTile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;

    ptx::launch_dependents();
    ptx::grid_dependency_wait();  // pass 1 complete

    // Exclusive prefix of destination counts over the earlier tiles.
    for (int d = warp; d < p.R; d += kWarps) {
        int sum = 0;
        for (int i = lane; i < tile; i += 32)
            sum += p.tile_counts[((size_t)s * p.ntiles + i) * p.RP + d];
        sum = warp_sum(sum);
        if (lane == 0) prefix[d] = sum;
    }

    // This CTA also finishes the experts e == cta (mod ncta) of the
    // local-expert histogram (sum of all tiles' partial counts).
    {
        const int ncta = p.R * p.ntiles, cta = s * p.ntiles + tile;
        for (int e = cta + warp * ncta; e < p.E; e += kWarps * ncta) {
            int sum = 0;
            for (int c = lane; c < ncta; c += 32) sum += p.tile_hist[(size_t)c * p.E + e];
            sum = warp_sum(sum);
            if (lane == 0) p.local_counts[e] = sum;
        }
    }

    const bool active = t < p.T;
    const uint32_t mask = active ? p.dmask[(size_t)s * p.T + t] : 0u;
    for (int d = 0; d < p.R; ++d) {
        const uint32_t b = __ballot_sync(kFull, (mask >> d) & 1u);
        if (lane == 0) warp_cnt[warp][d] = __popc(b);
    }
    __syncthreads();
    if (threadIdx.x < p.R) {
        const int d = threadIdx.x;
        int run = prefix[d];
        for (int w = 0; w < kWarps; ++w) {
            warp_off[w][d] = run;
            run += warp_cnt[w][d];
        }
        tile_total[d] = run;
    }
    __syncthreads();

    const size_t tok = (size_t)s * p.T + (active ? t : 0);
    const int32_t *ids = p.topk_ids + tok * K;
    const float *wts = p.topk_w + tok * K;
    constexpr int KR = KT > 0 ? KT : 1;
    int32_t id_r[KR];
    float w_r[KR];
    if (KT > 0 && active) {
#pragma unroll
        for (int k = 0; k < KR; ++k) {
            id_r[k] = ids[k];
            w_r[k] = wts[k];
        }
    }
    const uint32_t lt = lanemask_lt();
    int32_t *srow = p.send_slot + tok * p.RP;
    float *wrow = p.dest_weight + tok * p.RP;

    for (int d = 0; d < p.R; ++d) {
        const bool has = (mask >> d) & 1u;
        const uint32_t b = __ballot_sync(kFull, has);
        if (!active) continue;
        int32_t slot = -1;
        float wsum = 0.0f;
        if (has) {
            slot = warp_off[warp][d] + __popc(b & lt);
            const size_t row = ((size_t)d * p.R + s) * p.m + slot;
            p.src_token[row] = t;
            int32_t *rid = p.recv_ids + row * K;
            float *rw = p.recv_w + row * K;
            if constexpr (KT > 0 && KT % 4 == 0) {
#pragma unroll
                for (int k0 = 0; k0 < KT; k0 += 4) {
                    int4 iv;
                    float4 fv;
                    int32_t *ie = &iv.x;
                    float *fe = &fv.x;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e = id_r[k0 + q];
                        const bool local = e >= 0 && e < p.E && e / p.Epr == d;
                        ie[q] = local ? e : -1;
                        fe[q] = local ? w_r[k0 + q] : 0.0f;
                        if (local) wsum = __fadd_rn(wsum, w_r[k0 + q]);
                    }
                    reinterpret_cast<int4 *>(rid)[k0 / 4] = iv;
                    reinterpret_cast<float4 *>(rw)[k0 / 4] = fv;
                }
            } else if constexpr (KT > 0) {
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    const int e = id_r[k];
                    const bool local = e >= 0 && e < p.E && e / p.Epr == d;
                    rid[k] = local ? e : -1;
                    rw[k] = local ? w_r[k] : 0.0f;
                    if (local) wsum = __fadd_rn(wsum, w_r[k]);
                }
            } else {
                for (int k = 0; k < K; ++k) {
                    const int e = ids[k];
                    const float wk = wts[k];
                    const bool local = e >= 0 && e < p.E && e / p.Epr == d;
                    rid[k] = local ? e : -1;
                    rw[k] = local ? wk : 0.0f;
                    if (local) wsum = __fadd_rn(wsum, wk);
                }
            }
        }
        srow[d] = slot;
        wrow[d] = wsum;
    }
    if (active) {
        for (int d = p.R; d < p.RP; ++d) {
            srow[d] = -1;
            wrow[d] = 0.0f;
        }
    }

    if (tile == p.ntiles - 1 && threadIdx.x < p.R)
        p.recv_counts[threadIdx.x * p.R + s] = tile_total[threadIdx.x];
}

template <typename Kern, typename P>
cudaError_t launch2d(Kern kern, const P &p, int ntiles, int R, size_t smem, cudaStream_t st,
                     bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ntiles, R, 1);
    cfg.blockDim = dim3(kRouteTile, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_route_count(const RouteCountParams &p, cudaStream_t st) {
    const size_t smem = (size_t)p.E * sizeof(int32_t);
    switch (p.K) {
        case 2: return launch2d(route_count_kernel<2>, p, p.ntiles, p.R, smem, st, false);
        case 4: return launch2d(route_count_kernel<4>, p, p.ntiles, p.R, smem, st, false);
        case 8: return launch2d(route_count_kernel<8>, p, p.ntiles, p.R, smem, st, false);
        default: return launch2d(route_count_kernel<0>, p, p.ntiles, p.R, smem, st, false);
    }
}

cudaError_t launch_route_scan(const RouteScanParams &p, cudaStream_t st, bool pdl) {
    switch (p.K) {
        case 2: return launch2d(route_scan_kernel<2>, p, p.ntiles, p.R, 0, st, pdl);
        case 4: return launch2d(route_scan_kernel<4>, p, p.ntiles, p.R, 0, st, pdl);
        case 8: return launch2d(route_scan_kernel<8>, p, p.ntiles, p.R, 0, st, pdl);
        default: return launch2d(route_scan_kernel<0>, p, p.ntiles, p.R, 0, st, pdl);
    }
}

}  // namespace moe
