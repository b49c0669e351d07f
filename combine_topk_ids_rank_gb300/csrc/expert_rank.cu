// expert_rank.cu -- the expert-side product on the rank planes: the pair
// lists that feed the gathered tcgen05 product (expert_gemm.cu) and the
// gated sum of each received row's expert outputs.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs", "Why": each expert applies its weights to the
// rows it received; vLLM applies the gates in the MoE layer).  A received
// row (d, s, j) carries one token and, in recv_topk_ids, the token's experts
// that live on rank d (-1 elsewhere).  Readings: expert e_k's output on the
// row is bf16 (the product of expert_gemm.cu), and rank d's message is
//   out[d][s][j][n] = bf16_rn( sum over k ascending with a local id of
//                              g_k * y_k[n] ),  g_k = recv_topk_w or 1,
// in binary32 from +0.0, one multiply and one add per term (no FMA).
//
// GB300 design:
//   * rank_pairs: one (row, k) pair per local id.  Every CTA forms the
//     exclusive prefix of the experts' pair counts (local_expert_counts of
//     the dispatch) in shared memory; each thread walks received rows and
//     places its pairs with one atomic per expert and warp (lanes naming
//     the same expert are grouped with a match), writing the pair's
//     receive row (expert-major, what the product gathers) and the pair
//     index of (row, k) (what the sum reads).  The order of pairs inside an
//     expert is not fixed; every pair's product is the same whatever its
//     place in a tile, and the sum runs over k in a fixed order.
//   * rows with one local expert (one pair) get their message straight from
//     the product's epilogue, bf16(+0 + g * bf16(y)) -- the same arithmetic
//     (rank_pairs marks such a pair with bit 31 of its row and keeps its gate).
//   * rank_pairs also lists the rows with several local experts (one
//     atomic per warp), so that the sum touches those rows only.
//   * rank_aggregate: one CTA per listed row at a time, each thread a few
//     16-byte vectors of the output row; the row's pairs are taken in
//     ascending k, their bf16 outputs widened and summed in fp32 registers,
//     the message stored as bf16.  An HBM stream: those pairs x N x 2 bytes
//     read, those rows x N x 2 bytes written; nothing else is read.
#include "expert.h"
#include "kernels.h"

#include "moe_a2a.h"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPairThreads = 256;
constexpr int kAggThreads = 128;  // threads on one output row
constexpr int kAggVec = 4;        // 16-byte vectors a thread has in flight per pair

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(kPairThreads) rank_pairs_kernel(const RankPairsParams p) {
    __shared__ int32_t pbase[kMaxExpertsExpertLayout + 1];
    __shared__ int32_t wsum[kPairThreads / 32];
    // exclusive prefix of the pair counts, 256 experts per step
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += kPairThreads) {
        const int e = e0 + (int)threadIdx.x;
        const int c = e < p.E ? __ldg(p.pair_counts + e) : 0;
        int v = c;  // inclusive scan inside the warp
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) wsum[warp] = v;
        __syncthreads();
        int before = carry;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        if (e < p.E) pbase[e] = before + v - c;
        int total = 0;
        for (int w = 0; w < kPairThreads / 32; ++w) total += wsum[w];
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) pbase[p.E] = carry;
    __syncthreads();

    const long long rows = (long long)p.R * p.R * p.m;
    const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long step = (long long)gridDim.x * blockDim.x;
    const uint32_t lt = lanemask_lt();
    // whole warps iterate together (the match and the shuffles need them)
    for (long long base = first - (threadIdx.x & 31); base < rows; base += step) {
        const long long row = base + (threadIdx.x & 31);
        bool live = row < rows;
        if (live) {
            const long long plane = row / p.m;
            const int j = (int)(row - plane * p.m);
            live = j < __ldg(p.recv_counts + plane);
        }
        int n_local = 0;  // a row with one local expert gets its message from the product
        if (live)
            for (int k = 0; k < p.K; ++k) n_local += __ldg(p.recv_ids + row * p.K + k) >= 0;
        {  // rows with several local experts: on the list the gated sum walks
            const uint32_t many = __ballot_sync(kFull, n_local >= 2);
            if (many != 0) {
                const int leader = __ffs(many) - 1;
                int at = 0;
                if ((int)(threadIdx.x & 31) == leader) at = atomicAdd(p.cursor + p.E, __popc(many));
                at = __shfl_sync(kFull, at, leader) + __popc(many & lt);
                if (n_local >= 2) {
                    if (at < p.multi_cap) p.multi[at] = (int32_t)row;
                    else atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);  // guard: never expected
                }
            }
        }
        for (int k = 0; k < p.K; ++k) {
            const int e = live ? __ldg(p.recv_ids + row * p.K + k) : -1;
            const uint32_t want = __ballot_sync(kFull, e >= 0);
            int pos = -1;
            if (want != 0) {
                const uint32_t same = __match_any_sync(kFull, e);
                if (e >= 0) {
                    const int leader = __ffs(same) - 1;
                    int got = 0;
                    if ((int)(threadIdx.x & 31) == leader)
                        got = atomicAdd(p.cursor + e, __popc(same));
                    got = __shfl_sync(same, got, leader);
                    pos = pbase[e] + got + __popc(same & lt);
                    if (pos < pbase[e + 1]) {
                        p.pair_row[pos] = (int32_t)((uint32_t)row | (n_local == 1 ? 0x80000000u : 0u));
                        if (n_local == 1)
                            p.pair_gate[pos] = p.apply_gates ? __ldg(p.recv_w + row * p.K + k)
                                                             : 1.0f;
                    } else {  // guard: more pairs than the dispatch counted
                        atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                        pos = -1;
                    }
                }
            }
            if (live) p.pair_of[row * p.K + k] = pos;
        }
    }
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

__global__ void __launch_bounds__(kAggThreads) rank_aggregate_kernel(const RankPairsParams p) {
    const int N8 = p.N / 8;
    const uint4 *y = reinterpret_cast<const uint4 *>(p.y);
    uint4 *out = reinterpret_cast<uint4 *>(p.out);
    __shared__ int s_pr[kMaxTopK];  // the row's pairs in ascending k
    __shared__ float s_g[kMaxTopK];  // and their gates
    __shared__ int s_n;
    long long rows = __ldg(p.cursor + p.E);
    if (rows > p.multi_cap) rows = p.multi_cap;  // (flagged by rank_pairs)
    for (long long i = blockIdx.x; i < rows; i += gridDim.x) {
        const long long row = __ldg(p.multi + i);
        if (threadIdx.x < 32) {  // K <= 32: one warp compacts the local slots
            const int k = threadIdx.x;
            const int q = k < p.K ? __ldg(p.pair_of + row * p.K + k) : -1;
            const uint32_t has = __ballot_sync(kFull, q >= 0);
            if (q >= 0) {
                const int at = __popc(has & lanemask_lt());
                s_pr[at] = q;
                s_g[at] = p.apply_gates ? __ldg(p.recv_w + row * p.K + k) : 1.0f;
            }
            if (k == 0) s_n = __popc(has);
        }
        __syncthreads();
        const int n = s_n;
        for (int c0 = threadIdx.x; c0 < N8; c0 += kAggThreads * kAggVec) {
            float a[kAggVec][8];
#pragma unroll
            for (int u = 0; u < kAggVec; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e) a[u][e] = 0.0f;
            for (int t = 0; t < n; ++t) {
                const long long pr = s_pr[t];
                const float g = s_g[t];
                uint4 v[kAggVec];
#pragma unroll
                for (int u = 0; u < kAggVec; ++u) {
                    const int c = c0 + u * kAggThreads;
                    v[u] = c < N8 ? __ldcs(y + pr * N8 + c) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kAggVec; ++u) {
                    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        a[u][2 * e] = __fadd_rn(a[u][2 * e], __fmul_rn(g, lo_f(w[e])));
                        a[u][2 * e + 1] = __fadd_rn(a[u][2 * e + 1], __fmul_rn(g, hi_f(w[e])));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kAggVec; ++u) {
                const int c = c0 + u * kAggThreads;
                if (c < N8)
                    __stcs(out + row * N8 + c,
                           make_uint4(pack_bf16x2(a[u][0], a[u][1]), pack_bf16x2(a[u][2], a[u][3]),
                                      pack_bf16x2(a[u][4], a[u][5]), pack_bf16x2(a[u][6], a[u][7])));
            }
        }
        __syncthreads();  // the next row's pairs replace these
    }
}

}  // namespace

cudaError_t launch_rank_pairs(const RankPairsParams &p, int num_sms, cudaStream_t st) {
    if (p.E > kMaxExpertsExpertLayout || p.K < 1 || p.K > kMaxTopK) return cudaErrorInvalidValue;
    const long long rows = (long long)p.R * p.R * p.m;
    long long grid = (rows + kPairThreads - 1) / kPairThreads;
    if (grid > 4LL * num_sms) grid = 4LL * num_sms;
    if (grid < 1) return cudaSuccess;
    rank_pairs_kernel<<<(unsigned)grid, kPairThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rank_aggregate(const RankPairsParams &p, int num_sms, cudaStream_t st) {
    if (p.N % 8 != 0 || p.K > kMaxTopK) return cudaErrorInvalidValue;
    // the number of listed rows is on the device: a persistent grid, one
    // row per CTA at a time (at most as many CTAs as the list can hold)
    long long grid = 8LL * num_sms;
    if (grid > p.multi_cap) grid = p.multi_cap;
    if (grid < 1) return cudaSuccess;
    rank_aggregate_kernel<<<(unsigned)grid, kAggThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
