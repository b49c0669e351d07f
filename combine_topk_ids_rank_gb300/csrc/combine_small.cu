// combine_small.cu -- the combine for small batches: each token's row split
// over a cluster of CTAs, every message of the token in flight at once.
//
// Operation: the same as combine.cu / combine_ring.cu (InferenceX PR #2450,
// "CollectiveX: add FlashInfer one-sided NVLink EP for the GB SKUs", "Kernel
// arithmetic read from source" and "Update -- the correctness failures are
// resolved"; vLLM PR #41382; magik.net "Fusing the Allreduce ...", "The
// Message Itself"):
//   acc[h] = sum over the token's destinations, ascending, of v or w * v in
//            fp32 from +0.0, no FMA;
//   unfused: out = bf16_rn(acc)
//   fused:   hsum = acc + residual; residual_out = bf16_rn(hsum);
//            out = bf16_rn(hsum * rsqrt(mean(hsum^2) + eps) * gamma)
//
// GB300 design, for batches too small to keep the persistent combines busy
// (their CTAs take one or two tokens in turn, each waiting for a few row
// round trips): one cluster of kClusterCtas CTAs per token, CTA r owning
// column slice r of the row.  Each warp reads the token's send row (lane =
// destination), then every thread issues the loads of its vectors of ALL
// the token's messages (in groups of 8, each group's loads issued before it
// is summed, in ascending order), so a token costs about one row round trip.
// The residual and gamma slices are requested first (inputs of the call,
// before the programmatic-launch wait).  The fused epilogue's sum of
// squares is a warp shuffle, a pass through shared memory, and an exchange
// of the cluster's partial sums through distributed shared memory (summed
// in cluster-rank order, so every CTA of the token gets the same total).
#include "kernels.h"
#include "ptx.cuh"

#include "moe_a2a.h"

#include <cooperative_groups.h>
#include <cuda_bf16.h>

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kGroup = 8;  // message rows whose loads are in flight together

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                      pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
}

template <bool WEIGHTED>
__device__ __forceinline__ void accumulate8(float (&a)[8], const uint4 v, const float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = lo_f(u[i]), hi = hi_f(u[i]);
        if (WEIGHTED) {
            a[2 * i] = __fadd_rn(a[2 * i], __fmul_rn(w, lo));
            a[2 * i + 1] = __fadd_rn(a[2 * i + 1], __fmul_rn(w, hi));
        } else {
            a[2 * i] = __fadd_rn(a[2 * i], lo);
            a[2 * i + 1] = __fadd_rn(a[2 * i + 1], hi);
        }
    }
}

template <int VPT, bool WEIGHTED, bool FUSED>
__global__ void __launch_bounds__(kSmallCombineMaxThreads)
    combine_small_kernel(const CombineParams p, const int cols8) {
    __shared__ float red[kSmallCombineMaxThreads / 32];
    __shared__ float parts[kClusterCtas];  // every CTA's sum of squares, pushed by each
    cg::cluster_group cluster = cg::this_cluster();
    // This CTA has started: the arrival half of a split cluster barrier,
    // waited on just before the partial sums are pushed into the other
    // CTAs' shared memory (which needs every CTA of the cluster running).
    if constexpr (FUSED) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int crank = (int)cluster.block_rank(), csize = (int)cluster.num_blocks();
    const long long i = blockIdx.x / csize;  // the token of this cluster

    int s, t;
    token_of(p.map, p.R, i, s, t);
    const long long tok = (long long)s * p.map.stride + t;
    const long long row0 = tok * p.H8;
    const int c0 = crank * cols8;  // this CTA's column slice (16-byte vectors)
    const int c1 = min(p.H8, c0 + cols8);

    const uint4 *eo = reinterpret_cast<const uint4 *>(p.expert_out);
    const uint4 *res = reinterpret_cast<const uint4 *>(p.residual);
    const uint4 *gam = reinterpret_cast<const uint4 *>(p.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(p.out);
    uint4 *rout = reinterpret_cast<uint4 *>(p.residual_out);

    // inputs of the call first: the residual and gamma slices
    uint4 rv[FUSED ? VPT : 1], gv[FUSED ? VPT : 1];
    if constexpr (FUSED) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = c0 + tid + j * nthreads;
            rv[j] = c < c1 ? __ldcs(res + row0 + c) : make_uint4(0, 0, 0, 0);
            gv[j] = c < c1 ? __ldg(gam + c) : make_uint4(0, 0, 0, 0);
        }
    }
    ptx::grid_dependency_wait();  // the dispatch's send table and the experts' rows

    // lane d: the token's entry d of the send row (slot and weight)
    int slot = -1;
    float w = 0.0f;
    if (lane < p.dest.P) {
        slot = __ldg(p.send_slot + tok * p.dest.P + lane);
        if (WEIGHTED) w = __ldg(p.dest_weight + tok * p.dest.P + lane);
        if (slot >= 0) {
            if (dest_row(p.dest, p.R, p.m, lane, s, slot) < 0) {
                // guard: never produced by the routing pass
                if (warp == 0 && crank == 0) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                slot = -1;
            } else if (!((p.active >> dest_rank(p.dest, lane, slot)) & 1u)) {
                slot = -1;  // the rank is gone
            }
        }
    }

    float acc[VPT][8];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;

    uint32_t live = __ballot_sync(kFull, slot >= 0);  // ascending destinations
    while (live != 0) {
        int dq[kGroup];
        float wq[kGroup];
        uint4 v[kGroup][VPT];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
            dq[q] = live != 0 ? __ffs(live) - 1 : -1;
            if (live != 0) live &= live - 1;
            const int src = dq[q] < 0 ? 0 : dq[q];
            const int sq = __shfl_sync(kFull, slot, src);
            wq[q] = WEIGHTED ? __shfl_sync(kFull, w, src) : 1.0f;
            if (dq[q] >= 0) {
                const long long base = dest_row_checked(p.dest, p.R, p.m, dq[q], s, sq) * p.H8;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int c = c0 + tid + j * nthreads;
                    v[q][j] = c < c1 ? __ldcs(eo + base + c) : make_uint4(0, 0, 0, 0);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q)
            if (dq[q] >= 0) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) accumulate8<WEIGHTED>(acc[j], v[q][j], wq[q]);
            }
    }

    if constexpr (!FUSED) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = c0 + tid + j * nthreads;
            if (c < c1) __stcs(out + row0 + c, pack8(acc[j]));
        }
        return;
    } else {
        // hsum = acc + residual (fp32); residual_out; sum of squares
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            accumulate8<false>(acc[j], rv[j], 1.0f);
            const int c = c0 + tid + j * nthreads;
            if (c < c1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ss += acc[j][e] * acc[j][e];
                if (rout != nullptr) __stcs(rout + row0 + c, pack8(acc[j]));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float v = 0.0f;
        for (int k = 0; k < nwarps; ++k) v += red[k];
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // all CTAs started
        if (tid < csize) *cluster.map_shared_rank(&parts[crank], tid) = v;  // into CTA tid
        cluster.sync();  // every CTA's partial has arrived; nothing remote after this
        float total = 0.0f;
        for (int r = 0; r < csize; ++r) total += parts[r];  // ascending rank, as before
        const float inv = rsqrtf(total / (float)p.H + p.eps);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = c0 + tid + j * nthreads;
            if (c >= c1) continue;
            const uint32_t u[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
            float y[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                y[2 * k] = acc[j][2 * k] * inv * lo_f(u[k]);
                y[2 * k + 1] = acc[j][2 * k + 1] * inv * hi_f(u[k]);
            }
            __stcs(out + row0 + c, pack8(y));
        }
    }
}

template <int VPT, bool W, bool F>
cudaError_t launch_t(const CombineParams &p, const SmallCombineShape &sh, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.tokens * sh.cluster), 1, 1);
    cfg.blockDim = dim3(sh.threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sh.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, combine_small_kernel<VPT, W, F>, p, sh.cols8);
}

template <int VPT>
cudaError_t by_flags(bool w, bool f, const CombineParams &p, const SmallCombineShape &sh,
                     cudaStream_t st) {
    if (w && f) return launch_t<VPT, true, true>(p, sh, st);
    if (w) return launch_t<VPT, true, false>(p, sh, st);
    if (f) return launch_t<VPT, false, true>(p, sh, st);
    return launch_t<VPT, false, false>(p, sh, st);
}

}  // namespace

bool combine_small_shape(int H, SmallCombineShape *sh) {
    // kClusterCtas CTAs per token; each CTA's slice covered by 1 or 2
    // vectors per thread in at most kSmallCombineMaxThreads threads.
    const int H8 = H / 8;
    sh->cluster = kClusterCtas;
    sh->cols8 = (H8 + sh->cluster - 1) / sh->cluster;
    sh->vpt = sh->cols8 <= kSmallCombineMaxThreads ? 1 : 2;
    const int th = (sh->cols8 + sh->vpt - 1) / sh->vpt;
    sh->threads = (th + 31) / 32 * 32;
    return sh->threads <= kSmallCombineMaxThreads;
}

cudaError_t launch_combine_small(const CombineParams &p, bool weighted, bool fused,
                                 const SmallCombineShape &sh, cudaStream_t st) {
    if (p.tokens < 1) return cudaSuccess;
    if (p.dest.P > 32 || p.out == nullptr) return cudaErrorInvalidValue;
    return sh.vpt == 1 ? by_flags<1>(weighted, fused, p, sh, st)
                       : by_flags<2>(weighted, fused, p, sh, st);
}

}  // namespace moe
