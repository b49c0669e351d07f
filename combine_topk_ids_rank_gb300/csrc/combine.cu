// combine.cu -- gather-sum of each token's per-rank messages, reduced once,
// with the optional fused residual add + RMSNorm epilogue.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs": "Kernel arithmetic read from source" -- fp32
// accumulation and a round-to-nearest-even bf16 store, no FMA in the store
// path; "Update -- the correctness failures are resolved" -- fp32
// accumulator with a single narrowing.  vLLM PR #41382 "[Bugfix] Fix double
// reduce ...": the combine output is already reduced.  magik.net "Fusing
// the Allreduce ...", "The Message Itself": reduction, residual add and
// RMSNorm in one kernel, saving a launch and a memory round trip):
//   acc[h] = sum over d in dmask(s,t), ascending d, of v or w(s,t,d) * v,
//            v = expert_out[d][s][slot(s,t,d)][h], fp32 from +0.0, no FMA
//   unfused: out = bf16_rn(acc)
//   fused:   hsum = acc + residual; residual_out = bf16_rn(hsum);
//            out = bf16_rn(hsum * rsqrt(mean(hsum^2) + eps) * gamma)
//
// GB300 design: one CTA per token row at a time, persistent over tokens.
// Each thread owns VPT 16-byte vectors (8 bf16) of the row, strided by the
// block so every warp load is 512 contiguous bytes.  Lane d of each warp
// holds the token's slot and weight for destination d (the next token's are
// loaded while the current one is summed); a ballot gives the live
// destinations, which are gathered in groups of G with all G rows' loads
// issued before the group is accumulated in ascending order, so G rows (plus
// the residual row) are in flight per CTA.  Loads and stores of the streamed rows bypass L1 and are
// marked evict-first; gamma stays in L1.  The mean of squares is a warp
// shuffle reduction followed by a cross-warp pass through shared memory.
#include "kernels.h"
#include "ptx.cuh"

#include "moe_a2a.h"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) { __stcs(p, v); }

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

// EXP: send-table entries are absolute rows of the expert layout (lane =
// top-k slot); otherwise slots of the (rank, source) planes (lane = rank).
template <int VPT, int G, bool WEIGHTED, bool FUSED, bool EXP>
__global__ void __launch_bounds__(kMaxThreads) combine_kernel(const CombineParams p) {
    __shared__ float red[2][kMaxThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;

    const uint4 *eo = reinterpret_cast<const uint4 *>(p.expert_out);
    const uint4 *res = reinterpret_cast<const uint4 *>(p.residual);
    const uint4 *gam = reinterpret_cast<const uint4 *>(p.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(p.out);
    uint4 *rout = reinterpret_cast<uint4 *>(p.residual_out);

    ptx::grid_dependency_wait();

    // Lane d of every warp holds destination d's slot and weight of a token;
    // the next token's are loaded while the current one is summed.
    auto load_route = [&](long long i, int &slot, float &w) {
        slot = -1;
        w = 0.0f;
        if (!EXP && i < p.tokens && lane < p.R && ((p.active >> lane) & 1u)) {
            int s, t;
            token_of(p.map, p.R, i, s, t);
            const long long tok = (long long)s * p.map.stride + t;
            slot = __ldg(p.send_slot + tok * p.RP + lane);
            if (WEIGHTED) w = __ldg(p.dest_weight + tok * p.RP + lane);
            if (slot >= p.m) {  // guard: never expected from the routing pass
                if (warp == 0) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                slot = -1;
            }
        } else if (EXP && i < p.tokens && lane < p.dest.P) {
            int s, t;
            token_of(p.map, p.R, i, s, t);
            const long long tok = (long long)s * p.map.stride + t;
            slot = __ldg(p.send_slot + tok * p.dest.P + lane);
            if (WEIGHTED) w = __ldg(p.dest_weight + tok * p.dest.P + lane);
            if (slot >= 0) {
                if (dest_row(p.dest, p.R, p.m, lane, s, slot) < 0) {
                    // guard: never expected from the routing pass
                    if (warp == 0) atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                    slot = -1;
                } else if (!((p.active >> dest_rank(p.dest, lane, slot)) & 1u)) {
                    slot = -1;  // the expert's rank is gone
                }
            }
        }
    };
    int slot_l, slot_n;
    float w_l, w_n;
    load_route(blockIdx.x, slot_l, w_l);

    int parity = 0;
    for (long long i = blockIdx.x; i < p.tokens; i += gridDim.x, parity ^= 1) {
        load_route(i + gridDim.x, slot_n, w_n);
        int s, t;
        token_of(p.map, p.R, i, s, t);
        const long long tok = (long long)s * p.map.stride + t;  // row of the token arrays
        const long long row0 = tok * p.H8;

        uint4 r[FUSED ? VPT : 1];
        if (FUSED) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = tid + j * nthreads;
                r[j] = v < p.H8 ? ld_stream(res + row0 + v) : make_uint4(0, 0, 0, 0);
            }
        }

        float acc[VPT][8];
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;

        // The token's destinations, ascending; up to G rows in flight at once.
        uint32_t live = __ballot_sync(kFull, slot_l >= 0);
        while (live != 0) {
            int dq[G], sq[G];
            float wq[G];
            uint4 v[G][VPT];
#pragma unroll
            for (int q = 0; q < G; ++q) {
                dq[q] = live != 0 ? __ffs(live) - 1 : -1;
                if (live != 0) live &= live - 1;
                const int src = dq[q] < 0 ? 0 : dq[q];
                sq[q] = __shfl_sync(kFull, slot_l, src);
                wq[q] = WEIGHTED ? __shfl_sync(kFull, w_l, src) : 1.0f;
                if (dq[q] >= 0) {
                    const long long base =
                        (EXP ? (long long)sq[q]
                             : ((long long)dq[q] * p.R + s) * p.m + sq[q]) * p.H8;
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const int c = tid + j * nthreads;
                        v[q][j] = c < p.H8 ? ld_stream(eo + base + c) : make_uint4(0, 0, 0, 0);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < G; ++q) {
                if (dq[q] >= 0) {
#pragma unroll
                    for (int j = 0; j < VPT; ++j) accumulate8<WEIGHTED>(acc[j], v[q][j], wq[q]);
                }
            }
        }
        slot_l = slot_n;
        w_l = w_n;

        if (!FUSED) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int c = tid + j * nthreads;
                if (c < p.H8) st_stream(out + row0 + c, pack8(acc[j]));
            }
            continue;
        }

        // hsum = acc + residual (fp32); residual_out; sum of squares.
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint32_t u[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[j][2 * i] = __fadd_rn(acc[j][2 * i], lo_f(u[i]));
                acc[j][2 * i + 1] = __fadd_rn(acc[j][2 * i + 1], hi_f(u[i]));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += acc[j][e] * acc[j][e];
            const int c = tid + j * nthreads;
            if (rout != nullptr && c < p.H8) st_stream(rout + row0 + c, pack8(acc[j]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        if (lane == 0) red[parity][warp] = ss;
        __syncthreads();
        float total = 0.0f;
        for (int i = 0; i < nwarps; ++i) total += red[parity][i];
        const float inv = rsqrtf(total / (float)(p.H) + p.eps);

#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = tid + j * nthreads;
            if (c >= p.H8) continue;
            const uint4 g = __ldg(gam + c);
            const uint32_t u[4] = {g.x, g.y, g.z, g.w};
            float y[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                y[2 * i] = acc[j][2 * i] * inv * lo_f(u[i]);
                y[2 * i + 1] = acc[j][2 * i + 1] * inv * hi_f(u[i]);
            }
            st_stream(out + row0 + c, pack8(y));
        }
    }
}

template <int VPT, int G, bool W, bool F>
cudaError_t shape_of(int nthreads, int num_sms, LaunchShape *shape) {
    int per_sm = 0, per_sm_e = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, combine_kernel<VPT, G, W, F, false>, nthreads, 0);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm_e, combine_kernel<VPT, G, W, F, true>, nthreads, 0);
    per_sm = per_sm_e < per_sm ? per_sm_e : per_sm;  // one shape serves both layouts
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    shape->grid = num_sms * per_sm;
    shape->block = nthreads;
    shape->smem = 0;
    return cudaSuccess;
}

template <int VPT, int G, bool W, bool F>
cudaError_t launch_t(const CombineParams &p, const LaunchShape &shape, cudaStream_t st) {
    long long grid = shape.grid;
    if (grid > p.tokens) grid = p.tokens;
    if (grid < 1) return cudaSuccess;
    if (p.dest.expert)
        return launch_pdl(combine_kernel<VPT, G, W, F, true>, dim3((unsigned)grid),
                          dim3(shape.block), 0, st, p);
    return launch_pdl(combine_kernel<VPT, G, W, F, false>, dim3((unsigned)grid),
                      dim3(shape.block), 0, st, p);
}

// Rows in flight per group: 8 while a thread holds at most 2 vectors of a
// row, else 4 (register budget).
template <int VPT>
constexpr int group_of() { return VPT <= 2 ? 8 : 4; }

template <int VPT>
cudaError_t dispatch_flags(bool weighted, bool fused, const CombineParams *p, int nthreads,
                           int num_sms, LaunchShape *shape, const LaunchShape *use,
                           cudaStream_t st) {
    constexpr int kGroup = group_of<VPT>();
    if (p == nullptr) {
        if (weighted && fused) return shape_of<VPT, kGroup, true, true>(nthreads, num_sms, shape);
        if (weighted) return shape_of<VPT, kGroup, true, false>(nthreads, num_sms, shape);
        if (fused) return shape_of<VPT, kGroup, false, true>(nthreads, num_sms, shape);
        return shape_of<VPT, kGroup, false, false>(nthreads, num_sms, shape);
    }
    if (weighted && fused) return launch_t<VPT, kGroup, true, true>(*p, *use, st);
    if (weighted) return launch_t<VPT, kGroup, true, false>(*p, *use, st);
    if (fused) return launch_t<VPT, kGroup, false, true>(*p, *use, st);
    return launch_t<VPT, kGroup, false, false>(*p, *use, st);
}

cudaError_t by_vpt(int vpt, bool weighted, bool fused, const CombineParams *p, int nthreads,
                   int num_sms, LaunchShape *shape, const LaunchShape *use, cudaStream_t st) {
    switch (vpt) {
        case 1: return dispatch_flags<1>(weighted, fused, p, nthreads, num_sms, shape, use, st);
        case 2: return dispatch_flags<2>(weighted, fused, p, nthreads, num_sms, shape, use, st);
        case 4: return dispatch_flags<4>(weighted, fused, p, nthreads, num_sms, shape, use, st);
        case 8: return dispatch_flags<8>(weighted, fused, p, nthreads, num_sms, shape, use, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t combine_prepare(int H, bool weighted, bool fused, int num_sms, LaunchShape *shape,
                            int *vpt) {
    const int H8 = H / 8;
    int v = 1;
    while (v < 8 && (H8 + v - 1) / v > kMaxThreads) v *= 2;
    int nthreads = (H8 + v - 1) / v;
    nthreads = (nthreads + 31) / 32 * 32;
    if (nthreads > kMaxThreads) return cudaErrorInvalidValue;
    *vpt = v;
    return by_vpt(v, weighted, fused, nullptr, nthreads, num_sms, shape, nullptr, nullptr);
}

cudaError_t launch_combine(const CombineParams &p, bool weighted, bool fused, int vpt,
                           const LaunchShape &shape, cudaStream_t st) {
    return by_vpt(vpt, weighted, fused, &p, shape.block, 0, nullptr, &shape, st);
}

}  // namespace moe
