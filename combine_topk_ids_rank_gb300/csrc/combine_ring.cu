// combine_ring.cu -- the combine with its row loads on the copy engine.
//
// Same operation as combine.cu (InferenceX PR #2450 "CollectiveX: add
// FlashInfer one-sided NVLink EP for the GB SKUs", "Kernel arithmetic read
// from source" and "Update -- the correctness failures are resolved":
// fp32 accumulation, one round-to-nearest-even narrowing; vLLM PR #41382:
// reduced exactly once; magik.net "Fusing the Allreduce ...", "The Message
// Itself": residual add + RMSNorm fused):
//   acc[h] = sum over d in dmask(s,t), ascending d, of v or w(s,t,d) * v
//   unfused: out = bf16_rn(acc)
//   fused:   hsum = acc + residual; residual_out = bf16_rn(hsum);
//            out = bf16_rn(hsum * rsqrt(mean(hsum^2) + eps) * gamma)
//
// GB300 design: persistent CTAs (two or more per SM), warp-specialised.
//   * The producer warp walks the CTA's tokens, reads each token's send
//     row (slot per destination, prefetched one token ahead), publishes a
//     token descriptor (row count and per-row weights, ascending rank) and
//     streams the token's residual row and message rows into a ring of
//     shared-memory row buffers with 1-D bulk asynchronous copies, each
//     completing on the buffer's "full" mbarrier.
//   * Consumer warps own 16-byte vectors of the row.  For every token they
//     take the rows in ring order (residual first, then messages in
//     ascending rank), accumulate in fp32 registers, release each buffer on
//     its "empty" mbarrier, and finish the epilogue: the mean of squares
//     is a warp shuffle reduction and a cross-warp pass through shared
//     memory synchronised by an mbarrier; outputs are stored directly.
// The ring is shallow (~48 KB, three rows at H=7168) so that several CTAs
// share an SM: each has a token in its epilogue while the others' rows are
// in flight, and the copy engine keeps the loads going independently of
// registers.  Every wait
// is bounded: on time-out the warp raises the timeout flag and stops, and
// the producer waits (bounded) for its copies still landing before exit.
#include "kernels.h"
#include "ptx.cuh"
#include "smem_limit.h"
#include "fp8.cuh"
#include "f32x2.cuh"

#include "moe_a2a.h"

#include <cuda_bf16.h>

#include <cstdlib>
#include <type_traits>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kDesc = 8;                  // token descriptors in flight
constexpr int kMaxRingSlots = 32;
constexpr int kMaxConsumerWarps = 8;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr size_t kRingBytesTarget = 48 * 1024;

__host__ __device__ constexpr int consumer_warps_max(int vpt) {
    return vpt == 4 ? 7 : kMaxConsumerWarps;
}

struct TokenDesc {
    int32_t n;       // message rows of the token
    int32_t pad;
    float w[32];     // per-row weight, ascending destination rank
};

struct Ring {
    uint8_t *rows;
    uint64_t *full, *empty, *dfull, *dempty, *rbar;
    TokenDesc *desc;
    float *red;      // [2 parities][2 values][kMaxConsumerWarps]
};

__host__ __device__ inline size_t ring_stride(int row_bytes) {
    return ((size_t)row_bytes + 127) / 128 * 128;
}

__host__ __device__ inline size_t ring_smem_bytes(int row_bytes, int slots) {
    return ring_stride(row_bytes) * slots + sizeof(uint64_t) * (2 * slots + 2 * kDesc + 2) +
           sizeof(TokenDesc) * kDesc + sizeof(float) * 4 * kMaxConsumerWarps;
}

__device__ inline Ring carve(uint8_t *smem, int row_bytes, int slots) {
    Ring r;
    r.rows = smem;
    r.full = reinterpret_cast<uint64_t *>(smem + ring_stride(row_bytes) * slots);
    r.empty = r.full + slots;
    r.dfull = r.empty + slots;
    r.dempty = r.dfull + kDesc;
    r.rbar = r.dempty + kDesc;
    r.desc = reinterpret_cast<TokenDesc *>(r.rbar + 2);
    r.red = reinterpret_cast<float *>(r.desc + kDesc);
    return r;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                     ptx::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

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

// a[j] += w * v[j] (or v[j]), each product and sum rounded to binary32 (no
// FMA).  PACKED: the sums two lanes per instruction (identical results);
// used by the FP8-output combine at 4 or more vectors per thread.
// The products stay scalar: a paired multiply feeding a paired add was
// measured to come out fused (one rounding), which the sum must not be.
template <bool WEIGHTED, bool PACKED>
__device__ __forceinline__ void accumulate8(float (&a)[8], const uint4 v, const float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    if constexpr (PACKED) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const x2::f2 x = WEIGHTED ? x2::pack(__fmul_rn(w, lo_f(u[i])), __fmul_rn(w, hi_f(u[i])))
                                      : x2::bf16x2(u[i]);
            x2::unpack(x2::add(x2::pack(a[2 * i], a[2 * i + 1]), x), a[2 * i], a[2 * i + 1]);
        }
    } else {
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
}

// ---- producer warp ----------------------------------------------------------

template <bool WEIGHTED, bool FUSED>
__device__ void produce(const CombineParams &p, const Ring &r, int slots) {
    const int lane = threadIdx.x & 31;
    const uint8_t *eo = reinterpret_cast<const uint8_t *>(p.expert_out);
    const uint8_t *res = reinterpret_cast<const uint8_t *>(p.residual);
    const uint32_t row_bytes = 2u * (uint32_t)p.H;
    const size_t stride = ring_stride((int)row_bytes);
    const uint32_t lt = lanemask_lt();

    // the CTA's i-th token: its row in the token arrays and its source rank
    auto row_of = [&](long long i, int &s) -> long long {
        int t;
        token_of(p.map, p.R, i, s, t);
        return (long long)s * p.map.stride + t;
    };
    auto load_route = [&](long long i, int &slot, float &w) {
        slot = -1;
        w = 0.0f;
        if (i < p.tokens && lane < p.dest.P) {
            int s;
            const long long tok = row_of(i, s);
            slot = __ldg(p.send_slot + tok * p.dest.P + lane);
            if (WEIGHTED) w = __ldg(p.dest_weight + tok * p.dest.P + lane);
            if (slot >= 0) {
                if (dest_row(p.dest, p.R, p.m, lane, s, slot) < 0) {
                    // guard: never expected from the routing pass
                    atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                    slot = -1;
                } else if (!((p.active >> dest_rank(p.dest, lane, slot)) & 1u)) {
                    slot = -1;  // the rank is gone
                }
            }
        }
    };

    uint32_t q = 0;  // rows issued
    int qb = 0;            // q mod slots, stepped with q
    uint32_t qph = 0;      // (q / slots) & 1
    bool ok = true;
    auto issue_row = [&](const uint8_t *src) -> bool {
        const int b = qb;
        if (!ptx::mbar_wait_bounded(&r.empty[b], qph ^ 1u, kWaitLimit)) return false;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&r.full[b], row_bytes);
            ptx::bulk_g2s(r.rows + b * stride, src, row_bytes, &r.full[b]);
        }
        ++q;
        if (++qb == slots) {
            qb = 0;
            qph ^= 1u;
        }
        return true;
    };

    int slot, slot_next;
    float w, w_next;
    long long i = blockIdx.x;
    load_route(i, slot, w);
    for (uint32_t j = 0; i < p.tokens; i += gridDim.x, ++j) {
        load_route(i + gridDim.x, slot_next, w_next);
        int s;
        const long long tok = row_of(i, s);
        const bool valid = slot >= 0;
        const uint32_t bal = __ballot_sync(kFull, valid);

        const int ds = j % kDesc;
        if (!ptx::mbar_wait_bounded(&r.dempty[ds], ((j / kDesc) & 1u) ^ 1u, kWaitLimit)) {
            ok = false;
            break;
        }
        if (valid) r.desc[ds].w[__popc(bal & lt)] = w;
        if (lane == 0) r.desc[ds].n = __popc(bal);
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.dfull[ds]);

        if (FUSED && !issue_row(res + tok * row_bytes)) {
            ok = false;
            break;
        }
        uint32_t b = bal;
        while (b != 0) {
            const int d = __ffs(b) - 1;
            b &= b - 1;
            const int sl = __shfl_sync(kFull, slot, d);
            const long long row = dest_row_checked(p.dest, p.R, p.m, d, s, sl);
            if (!issue_row(eo + row * row_bytes)) {
                ok = false;
                break;
            }
        }
        if (!ok) break;
        slot = slot_next;
        w = w_next;
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
        // Let the copies already issued land before the CTA's shared memory goes away.
        const uint32_t first = q > (uint32_t)slots ? q - slots : 0u;
        for (uint32_t k = first; k < q; ++k)
            ptx::mbar_wait_bounded(&r.full[k % slots], (k / slots) & 1u, kWaitLimit);
    }
}

// ---- consumer warps ---------------------------------------------------------

template <int VPT, bool WEIGHTED, bool FUSED, bool OUT8>
__device__ void consume(const CombineParams &p, const Ring &r, int slots, int ncw) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nct = ncw * 32;
    const size_t stride = ring_stride(2 * p.H);
    const uint4 *gam = reinterpret_cast<const uint4 *>(p.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(p.out);
    uint4 *rout = reinterpret_cast<uint4 *>(p.residual_out);

    // gamma stays in registers for the whole kernel where the row is short
    // enough (it is read once per token, on the epilogue's critical path)
    constexpr bool kGammaRegs = FUSED && VPT == 4;
    // Paired fp32 arithmetic where the FP8 output's extra per-element work
    // makes the kernel issue-bound (measured: FP8-output combine 432.7 ->
    // 413.4 us at prefill; no gain for the bf16 output, which stays scalar).
    constexpr bool kPacked = OUT8 && VPT >= 4;
    uint4 gv[kGammaRegs ? VPT : 1];
    if constexpr (kGammaRegs) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = tid + v * nct;
            gv[v] = c < p.H8 ? __ldg(gam + c) : make_uint4(0, 0, 0, 0);
        }
    }

    uint32_t q = 0, nred = 0;  // rows consumed, reductions done
    int qb = 0;                // q mod slots, stepped with q
    uint32_t qph = 0;          // (q / slots) & 1
    auto next_row = [&]() {
        ++q;
        if (++qb == slots) {
            qb = 0;
            qph ^= 1u;
        }
    };
    bool ok = true;
    // Over the CTA's consumer threads: the sum of `a` and, if TWO, the max of
    // `b` -- warp shuffles, then one slot per warp and value in shared
    // memory, synchronised by an mbarrier (two slot sets / barriers used
    // alternately).
    auto block_reduce = [&](auto two, float a, float b, float &ra, float &rb) -> bool {
        constexpr bool TWO = decltype(two)::value;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(kFull, a, o);
            if (TWO) b = fmaxf(b, __shfl_xor_sync(kFull, b, o));
        }
        float *red = r.red + (nred & 1) * 2 * kMaxConsumerWarps;
        uint64_t *bar = &r.rbar[nred & 1];
        if (lane == 0) {
            red[warp] = a;
            if (TWO) red[kMaxConsumerWarps + warp] = b;
            mbar_arrive(bar);
        }
        if (!ptx::mbar_wait_bounded(bar, (nred >> 1) & 1u, kWaitLimit)) return false;
        ++nred;
        ra = 0.0f;
        rb = 0.0f;
        for (int i = 0; i < ncw; ++i) {
            ra += red[i];
            if (TWO) rb = fmaxf(rb, red[kMaxConsumerWarps + i]);
        }
        return true;
    };
    using One = std::false_type;
    using Two = std::true_type;
    for (long long i = blockIdx.x, j = 0; i < p.tokens; i += gridDim.x, ++j) {
        int s, t;
        token_of(p.map, p.R, i, s, t);
        const long long tok = (long long)s * p.map.stride + t;
        const int ds = (int)(j % kDesc);
        if (!ptx::mbar_wait_bounded(&r.dfull[ds], (uint32_t)((j / kDesc) & 1), kWaitLimit)) {
            ok = false;
            break;
        }
        const int n = r.desc[ds].n;

        uint4 rv[FUSED ? VPT : 1];
        if (FUSED) {
            const int b = qb;
            if (!ptx::mbar_wait_bounded(&r.full[b], qph, kWaitLimit)) {
                ok = false;
                break;
            }
            const uint4 *row = reinterpret_cast<const uint4 *>(r.rows + b * stride);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = tid + v * nct;
                rv[v] = c < p.H8 ? row[c] : make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[b]);
            next_row();
        }

        float acc[VPT][8];
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[v][e] = 0.0f;

        for (int i = 0; i < n; ++i) {
            const float wi = WEIGHTED ? r.desc[ds].w[i] : 1.0f;
            const int b = qb;
            if (!ptx::mbar_wait_bounded(&r.full[b], qph, kWaitLimit)) {
                ok = false;
                break;
            }
            const uint4 *row = reinterpret_cast<const uint4 *>(r.rows + b * stride);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = tid + v * nct;
                if (c < p.H8) accumulate8<WEIGHTED, kPacked>(acc[v], row[c], wi);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[b]);
            next_row();
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.dempty[ds]);

        const long long row0 = tok * p.H8;
        if (!FUSED && !OUT8) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = tid + v * nct;
                if (c < p.H8) __stcs(out + row0 + c, pack8(acc[v]));
            }
            continue;
        }

        float amax = 0.0f;  // OUT8: max |value quantised| of the row
        if (FUSED) {
            // hsum = acc + residual (fp32); residual_out = bf16(hsum);
            // y = hsum * rsqrt(mean(hsum^2) + eps) * gamma.  With FP8 output
            // the kernel forms y = inv * (hsum * gamma): inv > 0 and
            // rounding is monotone, so max|y| = inv * max|hsum * gamma|
            // exactly and one reduction serves both the mean and the amax.
            float ss = 0.0f, gmax = 0.0f;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                accumulate8<false, kPacked>(acc[v], rv[v], 1.0f);  // + residual
#pragma unroll
                for (int e = 0; e < 8; ++e) ss += acc[v][e] * acc[v][e];
                const int c = tid + v * nct;
                if (rout != nullptr && c < p.H8) __stcs(rout + row0 + c, pack8(acc[v]));
                if (OUT8 && c < p.H8) {
                    const uint4 g = kGammaRegs ? gv[kGammaRegs ? v : 0] : __ldg(gam + c);
                    const uint32_t gu[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if constexpr (kPacked) {
                            x2::unpack(x2::mul(x2::pack(acc[v][2 * i], acc[v][2 * i + 1]),
                                               x2::bf16x2(gu[i])),
                                       acc[v][2 * i], acc[v][2 * i + 1]);
                        } else {
                            acc[v][2 * i] = __fmul_rn(acc[v][2 * i], lo_f(gu[i]));
                            acc[v][2 * i + 1] = __fmul_rn(acc[v][2 * i + 1], hi_f(gu[i]));
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) gmax = fmaxf(gmax, fabsf(acc[v][e]));
                }
            }
            float total, gtot;
            if (!block_reduce(std::integral_constant<bool, OUT8>(), ss, gmax, total, gtot)) {
                ok = false;
                break;
            }
            const float inv = rsqrtf(total / (float)p.H + p.eps);
            if (OUT8) {
                const x2::f2 inv2 = x2::pack(inv, inv);
#pragma unroll
                for (int v = 0; v < VPT; ++v)
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        x2::unpack(x2::mul(inv2, x2::pack(acc[v][e], acc[v][e + 1])), acc[v][e],
                                   acc[v][e + 1]);
                amax = __fmul_rn(inv, gtot);
            } else {
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int c = tid + v * nct;
                    if (c >= p.H8) continue;
                    const uint4 g = kGammaRegs ? gv[kGammaRegs ? v : 0] : __ldg(gam + c);
                    const uint32_t u[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[v][2 * i] = acc[v][2 * i] * inv * lo_f(u[i]);
                        acc[v][2 * i + 1] = acc[v][2 * i + 1] * inv * hi_f(u[i]);
                    }
                    __stcs(out + row0 + c, pack8(acc[v]));
                }
                continue;
            }
        } else {
            // FP8 output of the plain sum: amax of the fp32 accumulator
            float m = 0.0f;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = tid + v * nct;
                if (c < p.H8)
#pragma unroll
                    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(acc[v][e]));
            }
            float unused;
            if (!block_reduce(Two(), 0.0f, m, unused, amax)) {
                ok = false;
                break;
            }
        }

        // FP8 output: per-token scale amax / 448, e4m3 codes of value / scale
        const fp8::RowScale rs = fp8::row_scale(amax);
        uint2 *out8 = reinterpret_cast<uint2 *>(p.out8 + tok * (long long)p.H);
        uint2 codes[VPT];
        fp8::quantize_row<VPT>(acc, rs, codes);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = tid + v * nct;
            if (c < p.H8) __stcs(out8 + c, codes[v]);
        }
        if (tid == 0) p.out_scale[tok] = rs.s;
    }
    if (!ok && lane == 0) atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
}

template <int VPT, bool WEIGHTED, bool FUSED, bool OUT8>
__device__ __forceinline__ void ring_main(const CombineParams &p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int slots = p.ring_slots;
    const int ncw = (int)(blockDim.x >> 5) - 1;
    const Ring r = carve(smem, 2 * p.H, slots);
    if (threadIdx.x == 0) {
        for (int i = 0; i < slots; ++i) {
            ptx::mbar_init(&r.full[i], 1);
            ptx::mbar_init(&r.empty[i], ncw);
        }
        for (int i = 0; i < kDesc; ++i) {
            ptx::mbar_init(&r.dfull[i], 1);
            ptx::mbar_init(&r.dempty[i], ncw);
        }
        ptx::mbar_init(&r.rbar[0], ncw);
        ptx::mbar_init(&r.rbar[1], ncw);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::grid_dependency_wait();
    if ((int)(threadIdx.x >> 5) == ncw)
        produce<WEIGHTED, FUSED>(p, r, slots);
    else
        consume<VPT, WEIGHTED, FUSED, OUT8>(p, r, slots, ncw);
}

template <int VPT, bool WEIGHTED, bool FUSED, bool OUT8>
__global__ void __launch_bounds__((kMaxConsumerWarps + 1) * 32)
    combine_ring_kernel(const CombineParams p) {
    ring_main<VPT, WEIGHTED, FUSED, OUT8>(p);
}

// Four vectors per thread (4096 < H <= 7168): at most 7 consumer warps, so
// that two CTAs of 8 warps per SM leave 128 registers per thread (4 warps
// per SM sub-partition) and gamma fits in registers beside the accumulators.
template <bool WEIGHTED, bool FUSED, bool OUT8>
__global__ void __launch_bounds__((consumer_warps_max(4) + 1) * 32, 2)
    combine_ring_kernel_v4(const CombineParams p) {
    ring_main<4, WEIGHTED, FUSED, OUT8>(p);
}

template <int VPT, bool W, bool F, bool O>
constexpr void (*ring_kernel())(CombineParams) {
    if constexpr (VPT == 4) return combine_ring_kernel_v4<W, F, O>;
    else return combine_ring_kernel<VPT, W, F, O>;
}

template <int VPT, bool W, bool F, bool O>
cudaError_t launch_t(const CombineParams &p, const LaunchShape &shape, cudaStream_t st) {
    long long grid = shape.grid;
    if (grid > p.tokens) grid = p.tokens;
    if (grid < 1) return cudaSuccess;
    return launch_pdl(ring_kernel<VPT, W, F, O>(), dim3((unsigned)grid), dim3(shape.block),
                      shape.smem, st, p);
}

// One of three actions on the instantiation selected by (vpt, w, f, o):
// allow its dynamic shared memory, query its occupancy, or launch it.
enum class Act { Prepare, Occupancy, Launch };

template <int VPT, bool W, bool F, bool O>
cudaError_t act_t(Act a, const CombineParams *p, const LaunchShape &shape, cudaStream_t st,
                  int *per_sm) {
    switch (a) {
        case Act::Prepare:
            return raise_smem_limit(ring_kernel<VPT, W, F, O>(), shape.smem);
        case Act::Occupancy:
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                per_sm, ring_kernel<VPT, W, F, O>(), shape.block, shape.smem);
        default:
            return launch_t<VPT, W, F, O>(*p, shape, st);
    }
}

template <int VPT>
cudaError_t by_flags(Act a, bool w, bool f, bool o, const CombineParams *p,
                     const LaunchShape &shape, cudaStream_t st, int *per_sm) {
    const int k = (w ? 4 : 0) + (f ? 2 : 0) + (o ? 1 : 0);
    switch (k) {
        case 0: return act_t<VPT, false, false, false>(a, p, shape, st, per_sm);
        case 1: return act_t<VPT, false, false, true>(a, p, shape, st, per_sm);
        case 2: return act_t<VPT, false, true, false>(a, p, shape, st, per_sm);
        case 3: return act_t<VPT, false, true, true>(a, p, shape, st, per_sm);
        case 4: return act_t<VPT, true, false, false>(a, p, shape, st, per_sm);
        case 5: return act_t<VPT, true, false, true>(a, p, shape, st, per_sm);
        case 6: return act_t<VPT, true, true, false>(a, p, shape, st, per_sm);
        default: return act_t<VPT, true, true, true>(a, p, shape, st, per_sm);
    }
}

cudaError_t by_vpt(Act a, int vpt, bool w, bool f, bool o, const CombineParams *p,
                   const LaunchShape &shape, cudaStream_t st, int *per_sm) {
    switch (vpt) {
        case 1: return by_flags<1>(a, w, f, o, p, shape, st, per_sm);
        case 2: return by_flags<2>(a, w, f, o, p, shape, st, per_sm);
        case 4: return by_flags<4>(a, w, f, o, p, shape, st, per_sm);
        case 8: return by_flags<8>(a, w, f, o, p, shape, st, per_sm);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t combine_ring_prepare(int H, bool weighted, bool fused, bool out8, int num_sms,
                                 const Tuning &tn, LaunchShape *shape, int *vpt, int *slots) {
    const int H8 = H / 8;
    int v = 1;
    while (v < 8 && (H8 + v - 1) / v > consumer_warps_max(v) * 32) v *= 2;
    const int ncw = ((H8 + v - 1) / v + 31) / 32;
    if (ncw > consumer_warps_max(v)) return cudaErrorInvalidValue;
    int dev = 0, optin = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    // About 48 KB of ring per CTA (3 rows at H=7168): the residency of
    // several CTAs per SM (several tokens in the reduce/epilogue stage at
    // once) matters more than a deep ring; measured best on the prefill
    // shape (2-6 slots swept).  The FP8 output's longer epilogue wants rows
    // more in flight: 80 KB (5 rows; prefill 412.4 us at 3 rows, 397.1 at 4,
    // 393.7 at 5, where 4 rows made the bf16 output slower).  So does the
    // plain sum, whose tokens carry more messages than the ring holds (wide
    // EP, 6.5 rows of 8 KB per token: 163.6 us at 10 rows against 171.7 at 6
    // and 166.6-167.7 for the register combine; 14 rows lose a CTA per SM).
    const size_t target = (out8 || !fused) ? 80 * 1024 : kRingBytesTarget;
    int s = (int)(target / ring_stride(2 * H));
    s = s < 2 ? 2 : (s > kMaxRingSlots ? kMaxRingSlots : s);
    if (tn.combine_ring_slots >= 2 && tn.combine_ring_slots <= kMaxRingSlots)
        s = tn.combine_ring_slots;
    while (s > 2 && ring_smem_bytes(2 * H, s) > (size_t)optin) --s;
    if (ring_smem_bytes(2 * H, s) > (size_t)optin) return cudaErrorInvalidValue;
    *vpt = v;
    *slots = s;
    shape->block = (ncw + 1) * 32;
    shape->smem = ring_smem_bytes(2 * H, s);
    err = by_vpt(Act::Prepare, v, weighted, fused, out8, nullptr, *shape, nullptr, nullptr);
    if (err != cudaSuccess) return err;
    int per_sm = 1;
    err = by_vpt(Act::Occupancy, v, weighted, fused, out8, nullptr, *shape, nullptr, &per_sm);
    if (err != cudaSuccess) return err;
    shape->grid = num_sms * (per_sm < 1 ? 1 : per_sm);
    return cudaSuccess;
}

cudaError_t launch_combine_ring(const CombineParams &p, bool weighted, bool fused, bool out8,
                                int vpt, const LaunchShape &shape, cudaStream_t st) {
    return by_vpt(Act::Launch, vpt, weighted, fused, out8, &p, shape, st, nullptr);
}

}  // namespace moe
