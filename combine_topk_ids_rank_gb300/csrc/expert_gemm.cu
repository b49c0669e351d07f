// expert_gemm.cu -- the expert-side consumer of the expert planes: one
// linear map per expert applied to the rows that expert received, on the
// tcgen05 tensor cores.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs", "Why": between dispatch and combine each
// expert applies its weights to the rows it received; vLLM applies the
// gates in the MoE layer around this product).  Reading: W_e is N x H,
// stored as a linear layer stores it (row n = the weights of output n):
//   y[e][j][n] = bf16_rn( sum_h x[e][j][h] * w[e][n][h] ),  j < recv_counts[e],
// products of bf16 values accumulated in fp32 (order of the tensor cores).
//
// GB300 design: one CTA per 128 x BN output tile of one expert; tiles that
// start past the expert's row count leave at once (the counts are read on
// the device, no host round trip).  Four warps:
//   warp 0, one thread: TMA producer -- 2-D tiled loads (128-byte swizzle)
//     of the A tile (128 rows x 64 of x) and the B tile (BN rows x 64 of W)
//     into a ring of shared-memory stages, completing on the stage's full
//     mbarrier;
//   warp 1, one thread: MMA issuer -- per stage four tcgen05.mma of
//     128 x BN x 16 (bf16 in, f32 accumulated in tensor memory), then a
//     tcgen05.commit that frees the stage; a final commit signals the
//     epilogue;
//   warp 2 owns the tensor-memory allocation (BN columns);
//   epilogue, all four warps: warp w reads tensor-memory lanes 32w..32w+31
//     (rows of the tile) 32 columns at a time, narrows to bf16 and stores the
//     rows below the expert's count.
// Every mbarrier wait is bounded in wall time; on a timeout the kernel
// raises the flag, lets its issued copies and products finish, frees
// tensor memory and returns.
#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#include "moe_a2a.h"

#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // bf16 elements per 128-byte swizzled row
constexpr int kThreads = 128;
constexpr uint64_t kWaitNs = 500ull * 1000 * 1000;  // 0.5 s of wall time per wait

template <int BN, int STAGES>
struct GemmSmem {
    static constexpr int kA = kBM * kBK * 2;  // bytes of an A stage
    static constexpr int kB = BN * kBK * 2;   // bytes of a B stage
    static constexpr int kTiles = STAGES * (kA + kB);
    // tiles (1024-aligned) + barriers + the tensor-memory slot, + 1024 for
    // aligning the dynamic shared memory base
    static constexpr int kBytes = kTiles + (2 * STAGES + 1) * 8 + 16 + 1024;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, const ExpertGemmParams p) {
    using L = GemmSmem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int issued_s, failed_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // tile -> (expert, row tile, column tile)
    const int nt_per = p.N / BN;
    const long long tile = blockIdx.x;
    const int e = (int)(tile / ((long long)p.mtiles * nt_per));
    const int rest = (int)(tile % ((long long)p.mtiles * nt_per));
    const int mt = rest / nt_per, nt = rest % nt_per;
    const int count = p.recv_counts[e];
    if (mt * kBM >= count) return;  // uniform: nothing allocated yet

    const uint32_t base = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
    uint8_t *a_tiles = smem;
    uint8_t *b_tiles = smem + STAGES * L::kA;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kTiles);
    uint64_t *empty = full + STAGES;
    uint64_t *done = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        ptx::fence_mbar_init();
        issued_s = 0;
        failed_s = 0;
    }
    if (warp == 2) tc::tmem_alloc(tmem_slot, BN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tmem_slot;

    const int KB = p.H / kBK;
    const int row0 = e * p.cap + mt * kBM;  // first row of the A tile
    const int wrow0 = e * p.N + nt * BN;    // first row of the B tile

    if (warp == 0 && lane == 0) {
        // producer
        int kb = 0;
        for (; kb < KB; ++kb) {
            const int s = kb % STAGES;
            if (kb >= STAGES &&
                !ptx::mbar_wait_timed(&empty[s], (uint32_t)((kb / STAGES - 1) & 1), kWaitNs)) {
                failed_s = 1;
                break;
            }
            ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)(L::kA + L::kB));
            tc::tma_load_2d(a_tiles + s * L::kA, &tmap_x, kb * kBK, row0, &full[s]);
            tc::tma_load_2d(b_tiles + s * L::kB, &tmap_w, kb * kBK, wrow0, &full[s]);
        }
        issued_s = kb;
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, BN);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % STAGES;
            if (!ptx::mbar_wait_timed(&full[s], (uint32_t)((kb / STAGES) & 1), kWaitNs)) {
                failed_s = 1;
                break;
            }
            tc::fence_after_sync();
            const uint64_t ad = tc::smem_desc_sw128(ptx::smem_u32(a_tiles + s * L::kA));
            const uint64_t bd = tc::smem_desc_sw128(ptx::smem_u32(b_tiles + s * L::kB));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)  // 16 bf16 = 32 bytes = 2 descriptor units
                tc::mma_bf16(taddr, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            tc::commit(&empty[s]);
        }
        tc::commit(done);  // arrives once every product issued above has completed
    }

    // epilogue
    const bool ok = ptx::mbar_wait_timed(done, 0, kWaitNs);
    __syncwarp();  // lane 0 of warps 0 and 1 rejoin before the warp-wide loads
    tc::fence_after_sync();
    const int r = mt * kBM + 32 * warp + lane;  // row of this thread within the expert
    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out);
    for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc::ld_32x32(taddr + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
        tc::wait_ld();
        if (ok && r < count) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                out + ((long long)e * p.cap + r) * p.N + (long long)nt * BN + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
                o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                dst[q] = o;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && (failed_s || !ok)) {
        atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
        // copies issued but never consumed must land before shared memory goes
        for (int kb = issued_s - STAGES < 0 ? 0 : issued_s - STAGES; kb < issued_s; ++kb)
            ptx::mbar_wait_timed(&full[kb % STAGES], (uint32_t)((kb / STAGES) & 1), kWaitNs);
    }
    __syncthreads();
    if (warp == 2) tc::tmem_dealloc(taddr, BN);
}

// ---- host: tensor maps -------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(ptr);
    });
    return fn;
}

// bf16 matrix of `rows` x `cols` (row-major, cols contiguous), boxes of
// box_rows x 64 with the 128-byte swizzle; rows past the end read as zero.
bool make_map(CUtensorMap *m, const void *base, long long rows, int cols, int box_rows) {
    EncodeTiled enc = encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES>
cudaError_t launch_t(const ExpertGemmParams &p, cudaStream_t st) {
    using L = GemmSmem<BN, STAGES>;
    CUtensorMap mx, mw;
    if (!make_map(&mx, p.x, (long long)p.E * p.cap, p.H, kBM) ||
        !make_map(&mw, p.w, (long long)p.E * p.N, p.H, BN))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(expert_gemm_kernel<BN, STAGES>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::kBytes);
    if (err != cudaSuccess) return err;
    const long long tiles = (long long)p.E * p.mtiles * (p.N / BN);
    if (tiles < 1) return cudaSuccess;
    expert_gemm_kernel<BN, STAGES><<<(unsigned)tiles, kThreads, L::kBytes, st>>>(mx, mw, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gemm(const ExpertGemmParams &p, cudaStream_t st) {
    if (p.H % kBK != 0 || p.H < kBK || p.N % 128 != 0 || p.N < 128 || p.cap < 1)
        return cudaErrorInvalidValue;
    if (p.N % 256 == 0) return launch_t<256, 4>(p, st);
    return launch_t<128, 6>(p, st);
}

}  // namespace moe
