// combine_tree.cu -- compatibility combine: the bf16 pairwise tree over
// top-k slots of FlashInfer's one-sided combine up to version 0.6.15.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs", comment "Update -- the correctness failures
// are resolved"): one accumulator per top-k slot held in bf16, each operand
// at its original top-k slot (duplicate-rank slots blanked in place), reduced
// by the pairwise tree (a0+a1)(a2+a3)(a4+a5)(a6+a7); (a0+a2)(a4+a6);
// (a0+a4), with a bf16 rounding after every add.  Slot k carries the message
// of rank topk_dest[s][t][k] (written by the routing pass), or zero.  K <= 8,
// padded with zero slots to a power of two P.  Unweighted, as that combine
// is.  The optional fused epilogue is the library's: hsum = tree + residual
// (fp32), residual_out = bf16(hsum), out = bf16(hsum * rsqrt(mean(hsum^2) +
// eps) * gamma).
//
// A compatibility path, not a throughput path: one CTA per token at a time,
// each thread a 16-byte vector of the row per iteration, the fp32 row sum
// kept in shared memory for the normalisation.
#include "kernels.h"
#include "ptx.cuh"
#include "smem_limit.h"

#include "moe_a2a.h"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16r(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}
__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                      pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
}

template <bool FUSED>
__global__ void __launch_bounds__(kThreads) combine_tree_kernel(const CombineTreeParams p) {
    extern __shared__ float hsum_row[];  // [H] (fused only)
    __shared__ int dest[8], slot[8];
    __shared__ float red[kThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x;
    const uint4 *eo = reinterpret_cast<const uint4 *>(p.expert_out);
    const uint4 *res = reinterpret_cast<const uint4 *>(p.residual);
    const uint4 *gam = reinterpret_cast<const uint4 *>(p.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(p.out);
    uint4 *rout = reinterpret_cast<uint4 *>(p.residual_out);

    ptx::grid_dependency_wait();
    for (long long i = blockIdx.x; i < p.tokens; i += gridDim.x) {
        int s, t;
        token_of(p.map, p.R, i, s, t);
        const long long tok = (long long)s * p.map.stride + t;
        if (tid < 8) {
            int d = tid < p.K ? p.topk_dest[tok * p.K + tid] : -1;
            if (d >= 0 && !((p.active >> d) & 1u)) d = -1;  // rank gone since dispatch
            int sl = d >= 0 ? p.send_slot[tok * p.RP + d] : -1;
            if (sl >= p.m) {  // guard: never expected from the routing pass
                atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                d = -1;
            }
            dest[tid] = d;
            slot[tid] = sl;
        }
        __syncthreads();

        float ss = 0.0f;
        const long long row0 = tok * p.H8;
        for (int c = tid; c < p.H8; c += nt) {
            float a[8][8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (dest[k] >= 0)
                    v = __ldcs(eo + (((long long)dest[k] * p.R + s) * p.m + slot[k]) * p.H8 + c);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a[k][2 * i] = lo_f(u[i]);
                    a[k][2 * i + 1] = hi_f(u[i]);
                }
            }
#pragma unroll
            for (int stride = 1; stride < 8; stride *= 2) {
                if (stride >= p.P) break;
#pragma unroll
                for (int k = 0; k + stride < 8; k += 2 * stride)
#pragma unroll
                    for (int e = 0; e < 8; ++e) a[k][e] = bf16r(a[k][e] + a[k + stride][e]);
            }
            if (!FUSED) {
                __stcs(out + row0 + c, pack8(a[0]));
                continue;
            }
            const uint4 r = __ldcs(res + row0 + c);
            const uint32_t u[4] = {r.x, r.y, r.z, r.w};
            float h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[2 * i] = __fadd_rn(a[0][2 * i], lo_f(u[i]));
                h[2 * i + 1] = __fadd_rn(a[0][2 * i + 1], hi_f(u[i]));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ss += h[e] * h[e];
                hsum_row[c * 8 + e] = h[e];
            }
            if (rout != nullptr) __stcs(rout + row0 + c, pack8(h));
        }
        if (FUSED) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
            if (lane == 0) red[warp] = ss;
            __syncthreads();
            float total = 0.0f;
            for (int i = 0; i < nt / 32; ++i) total += red[i];
            const float inv = rsqrtf(total / (float)p.H + p.eps);
            for (int c = tid; c < p.H8; c += nt) {
                const uint4 g = __ldg(gam + c);
                const uint32_t u[4] = {g.x, g.y, g.z, g.w};
                float y[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    y[2 * i] = hsum_row[c * 8 + 2 * i] * inv * lo_f(u[i]);
                    y[2 * i + 1] = hsum_row[c * 8 + 2 * i + 1] * inv * hi_f(u[i]);
                }
                __stcs(out + row0 + c, pack8(y));
            }
        }
        __syncthreads();  // dest/slot/red/hsum_row are reused by the next token
    }
}

}  // namespace

cudaError_t launch_combine_tree(const CombineTreeParams &p, int num_sms, cudaStream_t st) {
    if (p.K < 1 || p.K > 8) return cudaErrorInvalidValue;
    const bool fused = p.residual != nullptr;
    int nt = (p.H8 + 31) / 32 * 32;
    nt = nt > kThreads ? kThreads : nt;
    long long grid = (long long)num_sms * 4;
    if (grid > p.tokens) grid = p.tokens;
    if (grid < 1) return cudaSuccess;
    const size_t smem = fused ? (size_t)p.H * sizeof(float) : 0;
    if (fused) {
        cudaError_t err = raise_smem_limit(combine_tree_kernel<true>, smem);
        if (err != cudaSuccess) return err;
        return launch_pdl(combine_tree_kernel<true>, dim3((unsigned)grid), dim3(nt), smem, st, p);
    }
    return launch_pdl(combine_tree_kernel<false>, dim3((unsigned)grid), dim3(nt), 0, st, p);
}

}  // namespace moe
