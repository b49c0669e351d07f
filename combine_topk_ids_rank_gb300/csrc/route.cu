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
// Two passes over tiles of `tile` tokens (256 by default, 32..256, one token
// per thread) of one source rank, grid = tiles x R:
//   pass 1 (route_count): per-tile destination counts (warp ballots), the
//          expert histogram added into the source rank's accumulator (so
//          that only that source's tiles contend for an address), the
//          bad-id flag, and (when asked) each token's slots inside its
//          tile, which with the tile prefixes is all the row copy needs.
//          The last tile of a source to finish (atomic ticket after
//          a fence; nothing waits) scans that source's tile counts into
//          exclusive per-tile prefixes and writes its recv counts (a source
//          of one tile writes its zero prefix and counts without the ticket).
//   pass 2 (route_scan):  loads its tokens' ids and weights and rebuilds
//          their destination masks (while pass 1 still runs when chained
//          to it by programmatic dependent launch; beside the row copy, on
//          a second stream, otherwise), then adds its tile prefix to a warp-ballot /
//          cross-warp scan inside the tile to get each token's slot on
//          every destination; writes all routing outputs (send rows as
//          16-byte vectors); grid z splits the destinations into groups of
//          dg (4, or 1 so that small batches still spread over many CTAs);
//          copies its share of the histogram accumulator
//          to local_expert_counts and sets it back to zero for the next call.
// Both passes are O(T) in work and O(1) in cross-tile reads per CTA.
#include "kernels.h"
#include "ptx.cuh"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWarps = kRouteTile / 32;
constexpr int kScanChunk = 2048;  // ints staged per step of the tile scan

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// (magic: owner_magic(Epr), kernels.h)
__device__ __forceinline__ bool is_local(int e, int E, unsigned long long magic, int d) {
    return e >= 0 && e < E && owner_of(e, magic) == d;
}

// Destination rank of a valid expert on an active rank, else -1.
__device__ __forceinline__ int live_rank(int e, int E, unsigned long long magic,
                                         uint32_t active) {
    if (e < 0 || e >= E) return -1;
    const int d = owner_of(e, magic);
    return ((active >> d) & 1u) ? d : -1;
}

// KT > 0: top_k known at compile time (ids/weights held in registers);
// KT == 0: any top_k, read from global memory (L1) when needed.
template <int KT>
__global__ void __launch_bounds__(kRouteTile) route_count_kernel(const RouteCountParams p) {
    extern __shared__ int32_t hist[];  // [E]
    __shared__ int32_t warp_cnt[kMaxWarps][32];
    const int tile = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = p.tile >> 5;
    const int t = tile * p.tile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;

    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    for (int e = threadIdx.x; e < p.E; e += p.tile) hist[e] = 0;
    __syncthreads();

    uint32_t mask = 0;
    bool bad = false;
    if (t < p.map.count[s]) {
        const int32_t *ids = p.topk_ids + ((size_t)s * p.map.stride + t) * K;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int e = ids[k];
            if (e == -1) continue;
            if (e < -1 || e >= p.E) {
                bad = true;
                continue;
            }
            const int d = owner_of(e, p.epr_magic);
            if (!((p.active >> d) & 1u)) continue;  // expert on an inactive rank
            mask |= 1u << d;
            atomicAdd(&hist[e], 1);
        }
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
            for (int w = 0; w < nwarps; ++w) sum += warp_cnt[w][d];
        p.tile_counts[((size_t)s * p.ntiles + tile) * p.RP + d] = sum;
    }
    // Slots inside the tile (the tile's exclusive prefix, once known, turns
    // them into plane slots): the row copy needs nothing else, so it can
    // start as soon as this pass ends.
    if (p.local_slot != nullptr) {
        const uint32_t lt = lanemask_lt();
        const bool token = t < p.map.count[s];
        int32_t *lrow = p.local_slot + ((size_t)s * p.map.stride + (token ? t : 0)) * p.RP;
        for (int d0 = 0; d0 < p.RP; d0 += 4) {
            int4 v;
            int32_t *ve = &v.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int d = d0 + q;
                const bool has = d < p.R && ((mask >> d) & 1u);
                const uint32_t b = __ballot_sync(kFull, has);  // whole warp: converged
                int slot = -1;
                if (has) {
                    slot = __popc(b & lt);
                    for (int w = 0; w < warp; ++w) slot += warp_cnt[w][d];
                }
                ve[q] = slot;
            }
            if (token) *reinterpret_cast<int4 *>(lrow + d0) = v;
        }
    }
    int32_t *acc = p.hist_accum + (size_t)s * p.E;  // one accumulator per source rank
    for (int e = threadIdx.x; e < p.E; e += p.tile)
        if (hist[e] != 0) atomicAdd(&acc[e], hist[e]);

    if (p.ntiles == 1) {  // the source's only tile: its prefix is zero
        if (threadIdx.x < p.RP) p.tile_prefix[(size_t)s * p.RP + threadIdx.x] = 0;
        if (threadIdx.x < p.R) {
            int sum = 0;
            for (int w = 0; w < nwarps; ++w) sum += warp_cnt[w][threadIdx.x];
            p.recv_counts[threadIdx.x * p.R + s] = sum;
        }
        return;
    }

    // The last tile of this source to get here turns the tile counts into
    // exclusive prefixes.  Classic fence-then-ticket: no thread waits.
    __shared__ int last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&p.tile_ticket[s], 1) == p.ntiles - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Stage the source's tile counts through shared memory (the histogram
    // buffer, at least kScanChunk ints) in coalesced chunks; one thread per
    // destination turns each column into an exclusive running sum.
    int *buf = hist;
    const int chunk_tiles = kScanChunk / p.RP;
    const int32_t *src = p.tile_counts + (size_t)s * p.ntiles * p.RP;
    int32_t *dst = p.tile_prefix + (size_t)s * p.ntiles * p.RP;
    int carry = 0;
    for (int c0 = 0; c0 < p.ntiles; c0 += chunk_tiles) {
        const int nt = min(chunk_tiles, p.ntiles - c0);
        __syncthreads();
        for (int x = threadIdx.x; x < nt * p.RP; x += p.tile)
            buf[x] = __ldcg(src + (size_t)c0 * p.RP + x);
        __syncthreads();
        if (threadIdx.x < p.R) {
            for (int i = 0; i < nt; ++i) {
                const int v = buf[i * p.RP + threadIdx.x];
                buf[i * p.RP + threadIdx.x] = carry;
                carry += v;
            }
        }
        __syncthreads();
        for (int x = threadIdx.x; x < nt * p.RP; x += p.tile)
            dst[(size_t)c0 * p.RP + x] = buf[x];
    }
    if (threadIdx.x < p.R) p.recv_counts[threadIdx.x * p.R + s] = carry;
    if (threadIdx.x == 0) p.tile_ticket[s] = 0;  // ready for the next call
}

template <int KT>
__global__ void __launch_bounds__(kRouteTile) route_scan_kernel(const RouteScanParams p) {
    __shared__ int32_t prefix[32];
    __shared__ int32_t warp_cnt[kMaxWarps][32];
    __shared__ int32_t warp_off[kMaxWarps][32];
    const int tile = blockIdx.x, s = blockIdx.y, group = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = p.tile >> 5;
    const int t = tile * p.tile + threadIdx.x;
    const int K = KT > 0 ? KT : p.K;
    const bool active = t < p.map.count[s];
    // This CTA's destinations: [d_lo, d_lo + dg)
    const int d_lo = group * p.dg;

    ptx::launch_dependents();

    // Inputs first (they do not depend on pass 1): ids, weights, mask.
    const size_t tok = (size_t)s * p.map.stride + (active ? t : 0);
    const int32_t *ids = p.topk_ids + tok * K;
    const float *wts = p.topk_w + tok * K;
    constexpr int KR = KT > 0 ? KT : 1;
    int32_t id_r[KR];
    float w_r[KR];
    uint32_t mask = 0;
    if (active) {
        if constexpr (KT > 0) {
#pragma unroll
            for (int k = 0; k < KR; ++k) {
                id_r[k] = ids[k];
                w_r[k] = wts[k];
                const int d = live_rank(id_r[k], p.E, p.epr_magic, p.active);
                if (d >= 0) mask |= 1u << d;
            }
        } else {
            for (int k = 0; k < K; ++k) {
                const int d = live_rank(ids[k], p.E, p.epr_magic, p.active);
                if (d >= 0) mask |= 1u << d;
            }
        }
    }
    for (int d = 0; d < p.R; ++d) {
        const uint32_t b = __ballot_sync(kFull, (mask >> d) & 1u);
        if (lane == 0) warp_cnt[warp][d] = __popc(b);
    }

    ptx::grid_dependency_wait();  // pass 1 complete: prefixes and histogram

    if (threadIdx.x < p.R)
        prefix[threadIdx.x] = p.tile_prefix[((size_t)s * p.ntiles + tile) * p.RP + threadIdx.x];

    // This CTA owns the experts e == cta (mod ncta) of the histogram: sum
    // the per-source accumulators and leave them at zero for the next call.
    {
        const int ncta = p.R * p.ntiles * (int)gridDim.z;
        const int cta = (s * p.ntiles + tile) * (int)gridDim.z + group;
        for (int e = cta + (int)threadIdx.x * ncta; e < p.E; e += p.tile * ncta) {
            int sum = 0;
            for (int r0 = 0; r0 < p.R; r0 += 8) {  // 8 loads in flight at a time
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    v[u] = r0 + u < p.R ? __ldcg(p.hist_accum + (size_t)(r0 + u) * p.E + e) : 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) sum += v[u];
            }
            for (int r = 0; r < p.R; ++r) p.hist_accum[(size_t)r * p.E + e] = 0;
            p.local_counts[e] = sum;
        }
    }
    __syncthreads();
    if (threadIdx.x < p.R) {
        const int d = threadIdx.x;
        int run = prefix[d];
        for (int w = 0; w < nwarps; ++w) {
            warp_off[w][d] = run;
            run += warp_cnt[w][d];
        }
    }
    __syncthreads();

    // the rank whose message each top-k slot carries (first slot of a rank;
    // later slots of the same rank and invalid ids carry none)
    if (p.topk_dest != nullptr && active && group == 0) {
        int8_t *dst = p.topk_dest + tok * K;
        uint32_t seen = 0;
        for (int k = 0; k < K; ++k) {
            const int e = KT > 0 ? id_r[k < KR ? k : 0] : ids[k];
            const int d = live_rank(e, p.E, p.epr_magic, p.active);
            int8_t v = -1;
            if (d >= 0 && !((seen >> d) & 1u)) {
                v = (int8_t)d;
                seen |= 1u << d;
            }
            dst[k] = v;
        }
    }

    const uint32_t lt = lanemask_lt();
    int32_t *srow = p.send_slot + tok * p.RP;
    float *wrow = p.dest_weight + tok * p.RP;

    for (int d0 = d_lo; d0 < d_lo + p.dg; d0 += 4) {
        int4 sv;
        float4 wv;
        int32_t *se = &sv.x;
        float *we = &wv.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int d = d0 + q;
            if (q >= p.dg) break;  // fewer than 4 destinations per CTA
            const bool has = d < p.R && ((mask >> d) & 1u);
            const uint32_t b = __ballot_sync(kFull, has);
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
                        for (int u = 0; u < 4; ++u) {
                            const bool local = is_local(id_r[k0 + u], p.E, p.epr_magic, d);
                            ie[u] = local ? id_r[k0 + u] : -1;
                            fe[u] = local ? w_r[k0 + u] : 0.0f;
                            if (local) wsum = __fadd_rn(wsum, w_r[k0 + u]);
                        }
                        reinterpret_cast<int4 *>(rid)[k0 / 4] = iv;
                        reinterpret_cast<float4 *>(rw)[k0 / 4] = fv;
                    }
                } else if constexpr (KT > 0) {
#pragma unroll
                    for (int k = 0; k < KT; ++k) {
                        const bool local = is_local(id_r[k], p.E, p.epr_magic, d);
                        rid[k] = local ? id_r[k] : -1;
                        rw[k] = local ? w_r[k] : 0.0f;
                        if (local) wsum = __fadd_rn(wsum, w_r[k]);
                    }
                } else {
                    for (int k = 0; k < K; ++k) {
                        const int e = ids[k];
                        const float wk = wts[k];
                        const bool local = is_local(e, p.E, p.epr_magic, d);
                        rid[k] = local ? e : -1;
                        rw[k] = local ? wk : 0.0f;
                        if (local) wsum = __fadd_rn(wsum, wk);
                    }
                }
            }
            se[q] = slot;
            we[q] = wsum;
        }
        if (active) {
            if (p.dg == 4) {
                *reinterpret_cast<int4 *>(srow + d0) = sv;
                *reinterpret_cast<float4 *>(wrow + d0) = wv;
            } else {
                srow[d0] = sv.x;
                wrow[d0] = wv.x;
            }
        }
    }
}

template <typename Kern, typename P>
cudaError_t launch2d(Kern kern, const P &p, size_t smem, cudaStream_t st, bool pdl,
                     unsigned gz = 1) {
    if (p.tile < 32 || p.tile > kRouteTile || p.tile % 32 != 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ntiles, p.R, gz);
    cfg.blockDim = dim3(p.tile, 1, 1);
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

cudaError_t launch_route_count(const RouteCountParams &pc, cudaStream_t st) {
    RouteCountParams p = pc;
    p.epr_magic = owner_magic(p.Epr);
    const size_t smem = (size_t)(p.E > kScanChunk ? p.E : kScanChunk) * sizeof(int32_t);
    switch (p.K) {
        case 2: return launch2d(route_count_kernel<2>, p, smem, st, true);
        case 4: return launch2d(route_count_kernel<4>, p, smem, st, true);
        case 8: return launch2d(route_count_kernel<8>, p, smem, st, true);
        default: return launch2d(route_count_kernel<0>, p, smem, st, true);
    }
}

cudaError_t launch_route_scan(const RouteScanParams &pc, cudaStream_t st, bool pdl) {
    RouteScanParams p = pc;
    p.epr_magic = owner_magic(p.Epr);
    if ((p.dg != 1 && p.dg != 4) || p.RP % p.dg != 0) return cudaErrorInvalidValue;
    const unsigned gz = (unsigned)(p.RP / p.dg);
    switch (p.K) {
        case 2: return launch2d(route_scan_kernel<2>, p, 0, st, pdl, gz);
        case 4: return launch2d(route_scan_kernel<4>, p, 0, st, pdl, gz);
        case 8: return launch2d(route_scan_kernel<8>, p, 0, st, pdl, gz);
        default: return launch2d(route_scan_kernel<0>, p, 0, st, pdl, gz);
    }
}

}  // namespace moe
