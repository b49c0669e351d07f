// dispatch_fp8.cu -- dispatch with an FP8 row payload and a per-token scale,
// and the standalone FP8 row quantiser.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs", "The adapter": an FP8 dispatch carries a
// scale payload next to the row and is validated against the cast round
// trip).  Readings: OCP e4m3, per-token scale = amax_h |x_h| / 448 (binary32
// division; 1 for an all-zero row), q_h = e4m3_rn_satfinite(x_h / scale)
// (binary32 quotient):
//   recv_x8[d][s][slot(s,t,d)][:] = q(x[s][t]),  recv_scale[d][s][slot] = scale
// for every destination of the token; padding never written.
//
// GB300 design: persistent CTAs of up to 256 threads fitted to the row (128
// threads x 7 vectors at H = 7168), one token row at a time.
// One thread keeps the next few bf16 rows of the CTA in flight with 1-D bulk
// copies into a shared-memory ring (mbarrier completion, bounded waits);
// each thread takes VPT 16-byte vectors of the row into registers, the
// row's amax is a warp shuffle + one cross-warp step (the only CTA barrier
// per token, which also frees the stage for the next copy), and every
// thread quantises its own vectors (fp8.cuh: one reciprocal per row,
// FMA-refined quotients, two elements per paired-fp32 instruction) and
// writes 8 code bytes per vector straight to each
// destination row -- consecutive threads write consecutive 8-byte pieces,
// so each warp store covers 256 contiguous bytes.  The row is read once and
// written once per destination at half the bf16 bytes.
#include "kernels.h"
#include "ptx.cuh"
#include "smem_limit.h"
#include "fp8.cuh"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;          // at most; the launch fits the row (fit_threads)
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 8;
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = lo_f(u[k]);
        f[2 * k + 1] = hi_f(u[k]);
    }
}

template <int VPT>
__global__ void __launch_bounds__(kThreads, 3) dispatch_fp8_kernel(const DispatchFp8Params p) {
    extern __shared__ __align__(128) uint8_t smem[];  // p.stages bf16 rows
    __shared__ uint64_t full[kMaxStages];
    __shared__ long long rows[2][kMaxTopK];  // destination rows (-1: none)
    __shared__ float red[2][kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x, nw = nt >> 5;
    const int S = p.stages;
    const uint32_t row_bytes = (uint32_t)p.H * 2;
    const size_t stride = ((size_t)row_bytes + 127) / 128 * 128;

    // Token k of this CTA is i = blockIdx.x + k * gridDim.x; its row goes
    // to stage k % S.  Thread 0 keeps S rows in flight.
    auto issue = [&](long long k, int b) {  // b = k mod S
        const long long i = blockIdx.x + k * (long long)gridDim.x;
        if (i >= p.tokens) return;
        int s, t;
        token_of(p.map, p.R, i, s, t);
        ptx::mbar_arrive_expect_tx(&full[b], row_bytes);
        ptx::bulk_g2s(smem + b * stride, p.x + ((long long)s * p.map.stride + t) * p.H,
                      row_bytes, &full[b]);
    };
    if (tid == 0) {
        for (int b = 0; b < S; ++b) ptx::mbar_init(&full[b], 1);
        ptx::fence_mbar_init();
        for (int k = 0; k < S; ++k) issue(k, k);  // inputs: before the routing pass ends
    }
    __syncthreads();
    ptx::grid_dependency_wait();

    bool ok = true;
    long long k = 0;
    int b = 0;             // k mod S, stepped with k
    uint32_t phase = 0;    // (k / S) & 1
    for (long long i = blockIdx.x; i < p.tokens; i += gridDim.x, ++k) {
        const int par = (int)(k & 1);
        int s, t;
        token_of(p.map, p.R, i, s, t);
        const long long tok = (long long)s * p.map.stride + t;
        if (tid < p.dest.P) {
            int sl = p.send_slot[tok * p.dest.P + tid];
            if (sl >= 0 && p.tile_prefix != nullptr)  // tile-local slot + the tile's prefix
                sl += p.tile_prefix[((long long)s * p.ntiles + t / p.tile) * p.dest.P + tid];
            long long row = -1;
            if (sl >= 0) {
                row = dest_row(p.dest, p.R, p.m, tid, s, sl);
                if (row < 0)  // guard: never expected from the routing pass
                    atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
            }
            rows[par][tid] = row;
        }
        ok = ptx::mbar_wait_bounded(&full[b], phase, kWaitLimit);
        uint4 cur[VPT];
        const uint4 *row = reinterpret_cast<const uint4 *>(smem + b * stride);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = tid + j * nt;
            cur[j] = (ok && c < p.H8) ? row[c] : make_uint4(0, 0, 0, 0);
            const uint32_t u[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                amax = fmaxf(amax, fmaxf(fabsf(lo_f(u[e])), fabsf(hi_f(u[e]))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        if (lane == 0) red[par][warp] = amax;
        // One barrier per token.  It also releases stage b (every thread has
        // its vectors in registers) and makes the wait outcome collective.
        // red[] and rows[] alternate by token parity: no thread reaches the
        // barrier of token k+2 before all have passed that of k+1, i.e.
        // finished token k.
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        if (tid == 0) {
            ptx::fence_proxy_async_smem();
            issue(k + S, b);  // the stage just released
        }
        amax = red[par][0];
        for (int w = 1; w < nw; ++w) amax = fmaxf(amax, red[par][w]);
        const fp8::RowScale rs = fp8::row_scale(amax);

        float f[VPT][8];
#pragma unroll
        for (int j = 0; j < VPT; ++j) unpack8(cur[j], f[j]);
        uint2 q[VPT];
        fp8::quantize_row<VPT>(f, rs, q);
        for (int d = 0; d < p.dest.P; ++d) {
            const long long dst_row = rows[par][d];
            if (dst_row < 0) continue;
            uint2 *dst = reinterpret_cast<uint2 *>(p.recv_x8 + dst_row * p.H);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int c = tid + j * nt;
                if (c < p.H8) __stcs(dst + c, q[j]);
            }
            if (tid == 0) p.recv_scale[dst_row] = rs.s;
        }
        if (++b == S) {
            b = 0;
            phase ^= 1u;
        }
    }
    if (!ok && tid == 0) {
        atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
        // let the copies in flight land before the shared memory goes away
        for (long long j = k; j < k + S; ++j)
            if (blockIdx.x + j * (long long)gridDim.x < p.tokens)
                ptx::mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), kWaitLimit);
    }
}

// fp32 rows -> e4m3 codes + per-row scale; one CTA per row at a time.
template <int VPT>
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const float *x, long long rows,
                                                                 int H, uint8_t *q, float *scale) {
    __shared__ float red[2][kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H8 = H / 8, nt = blockDim.x, nw = nt >> 5;
    int par = 0;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x, par ^= 1) {
        const float4 *src = reinterpret_cast<const float4 *>(x + r * (long long)H);
        float v[VPT][8];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = tid + j * nt;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (c < H8) {
                a = __ldcs(src + 2 * c);
                b = __ldcs(src + 2 * c + 1);
            }
            v[j][0] = a.x, v[j][1] = a.y, v[j][2] = a.z, v[j][3] = a.w;
            v[j][4] = b.x, v[j][5] = b.y, v[j][6] = b.z, v[j][7] = b.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[j][e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        if (lane == 0) red[par][warp] = amax;
        __syncthreads();
        amax = red[par][0];
        for (int w = 1; w < nw; ++w) amax = fmaxf(amax, red[par][w]);
        const fp8::RowScale rs = fp8::row_scale(amax);
        uint2 *dst = reinterpret_cast<uint2 *>(q + r * (long long)H);
        uint2 codes[VPT];
        fp8::quantize_row<VPT>(v, rs, codes);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = tid + j * nt;
            if (c < H8) __stcs(dst + c, codes[j]);
        }
        if (tid == 0) scale[r] = rs.s;
    }
}

// Threads per CTA: 128 while a row fits in 8 vectors per thread, else the
// fewest whole warps that cover it with 8; every thread then takes VPT =
// ceil(H8 / threads) vectors (H = 7168: 128 threads x 7 vectors, no idle
// tail), so the per-token work (reduction, scale, routing reads, address
// arithmetic) is spread over as many elements per thread as the registers
// allow.
int fit_threads(int H8) {
    if (H8 <= 8 * 128) return 128;
    return ((H8 + 7) / 8 + 31) / 32 * 32;
}

// Ring depth and residency of the FP8 dispatch, once per handle.  Stages:
// about 42 KB of bf16 rows per CTA (3 rows at H = 7168), at least 2
// (Tuning::fp8_dispatch_stages overrides, 2..8).
template <int VPT>
cudaError_t prepare_t(int H, int num_sms, int stages_override, int *stages, LaunchShape *shape) {
    const int threads = fit_threads(H / 8);
    const size_t stride = ((size_t)H * 2 + 127) / 128 * 128;
    int S = (int)((42u << 10) / stride);
    if (stages_override > 0) S = stages_override;
    S = S < 2 ? 2 : (S > kMaxStages ? kMaxStages : S);
    const size_t smem = stride * S;
    cudaError_t err = raise_smem_limit(dispatch_fp8_kernel<VPT>, smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_fp8_kernel<VPT>,
                                                        threads, smem);
    if (err != cudaSuccess) return err;
    *stages = S;
    shape->grid = num_sms * (per_sm < 1 ? 1 : per_sm);
    shape->block = threads;
    shape->smem = smem;
    return cudaSuccess;
}

template <int VPT>
cudaError_t launch_t(const DispatchFp8Params &p, const LaunchShape &shape, cudaStream_t st) {
    long long grid = shape.grid;
    if (grid > p.tokens) grid = p.tokens;
    if (grid < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(shape.block, 1, 1);
    cfg.dynamicSmemBytes = shape.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_fp8_kernel<VPT>, p);
}

template <int VPT>
cudaError_t launch_q(const float *x, long long rows, int H, uint8_t *q, float *scale,
                     int num_sms, cudaStream_t st) {
    const int threads = fit_threads(H / 8);
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, quantize_rows_kernel<VPT>, threads, 0);
    if (err != cudaSuccess) return err;
    long long grid = (long long)num_sms * (per_sm < 1 ? 1 : per_sm);
    if (grid > rows) grid = rows;
    if (grid < 1) return cudaSuccess;
    quantize_rows_kernel<VPT><<<(unsigned)grid, threads, 0, st>>>(x, rows, H, q, scale);
    return cudaGetLastError();
}

int vectors_per_thread(int H8) {
    const int nt = fit_threads(H8);
    return (H8 + nt - 1) / nt;
}

// Instantiations for VPT = 1..8.
template <template <int> class F, typename... A>
cudaError_t by_vpt(int vpt, A... a) {
    switch (vpt) {
        case 1: return F<1>::run(a...);
        case 2: return F<2>::run(a...);
        case 3: return F<3>::run(a...);
        case 4: return F<4>::run(a...);
        case 5: return F<5>::run(a...);
        case 6: return F<6>::run(a...);
        case 7: return F<7>::run(a...);
        case 8: return F<8>::run(a...);
        default: return cudaErrorInvalidValue;
    }
}

template <int VPT>
struct DispatchPrepare {
    static cudaError_t run(int H, int num_sms, int stages_override, int *stages,
                           LaunchShape *shape) {
        return prepare_t<VPT>(H, num_sms, stages_override, stages, shape);
    }
};

template <int VPT>
struct DispatchLaunch {
    static cudaError_t run(const DispatchFp8Params *p, const LaunchShape *shape,
                           cudaStream_t st) {
        return launch_t<VPT>(*p, *shape, st);
    }
};

template <int VPT>
struct QuantLaunch {
    static cudaError_t run(const float *x, long long rows, int H, uint8_t *q, float *scale,
                           int num_sms, cudaStream_t st) {
        return launch_q<VPT>(x, rows, H, q, scale, num_sms, st);
    }
};

}  // namespace

cudaError_t dispatch_fp8_prepare(int H, int num_sms, const Tuning &tn, DispatchFp8Params *p,
                                 LaunchShape *shape) {
    if (H % 16 != 0 || H / 8 > 2048) return cudaErrorInvalidValue;
    return by_vpt<DispatchPrepare>(vectors_per_thread(H / 8), H, num_sms,
                                   tn.fp8_dispatch_stages, &p->stages, shape);
}

cudaError_t launch_dispatch_fp8(const DispatchFp8Params &p, const LaunchShape &shape,
                                cudaStream_t st) {
    if (p.H % 16 != 0 || p.H8 > 2048 || p.stages < 2) return cudaErrorInvalidValue;
    return by_vpt<DispatchLaunch>(vectors_per_thread(p.H8), &p, &shape, st);
}

cudaError_t launch_quantize_rows_fp8(const float *x, long long rows, int H, uint8_t *q,
                                     float *scale, int num_sms, cudaStream_t st) {
    if (H % 8 != 0 || H / 8 > 2048) return cudaErrorInvalidValue;
    return by_vpt<QuantLaunch>(vectors_per_thread(H / 8), x, rows, H, q, scale, num_sms, st);
}

}  // namespace moe
