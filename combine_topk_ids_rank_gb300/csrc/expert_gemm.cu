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
// GB300 design: a persistent kernel, one CTA per SM, over the useful
// 128 x BN output tiles only (tile list built in shared memory from the
// device-side row counts; raster: expert by expert, groups of row tiles
// (16 by default), column tile outer inside a group, so that concurrent CTAs
// share weight and row tiles in L2).  Six warps:
//   warp 4, one thread: TMA producer -- 2-D tiled loads (128-byte swizzle)
//     of the A tile (128 rows x 64 of x) and the B tile (BN rows x 64 of W)
//     into a ring of shared-memory stages that runs on across tiles;
//   warp 5: tensor-memory owner (2 x BN columns: two accumulators) and, one
//     thread, the MMA issuer -- per stage four tcgen05.mma of 128 x BN x 16
//     (bf16 in, f32 accumulated in tensor memory), a tcgen05.commit that
//     frees the stage, and one per tile that hands the accumulator over;
//   warps 0-3: epilogue -- warp w reads tensor-memory lanes 32w..32w+31 (rows
//     of the tile) 32 columns at a time, narrows to bf16, stores the rows
//     below the expert's count and frees the accumulator, while the MMA
//     thread already fills the other one.
// FP8 operands (either row source): e4m3 codes, 128 per stage row, products
// of .kind::f8f6f4 into the same fp32 accumulators; the epilogue multiplies
// by the A row's scale and the column's scale before the bf16 narrowing.
#include "expert.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#include "moe_a2a.h"

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;    // bytes of a stage row (one 128-byte swizzle span):
                                  // 64 bf16 or 128 e4m3 values
constexpr int kEpiWarps = 4;      // warps 0-3: epilogue (tensor-memory lane quadrants)
constexpr int kProducerWarp = 4;  // TMA
constexpr int kMmaWarp = 5;       // MMA issue + tensor-memory allocation
constexpr int kThreads = 6 * 32;
// Gathered rows (rank planes): warps 6-9 fetch the A tile, one thread per
// tile row, with 16-byte cp.async copies into the 128-byte-swizzled layout.
constexpr int kLoaderWarp0 = 6;
constexpr int kLoaderThreads = kBM;
constexpr int kThreadsGather = kThreads + kLoaderThreads;
constexpr uint64_t kWaitNs = 500ull * 1000 * 1000;  // 0.5 s of wall time per wait

template <int BN, int STAGES>
struct GemmSmem {
    static constexpr int kA = kBM * kRowBytes;  // bytes of an A stage
    static constexpr int kB = BN * kRowBytes;   // bytes of a B stage
    static constexpr int kTiles = STAGES * (kA + kB);
    // tiles (1024-aligned) + ring and accumulator barriers + the tensor-memory
    // slot, + 1024 for aligning the dynamic shared memory base
    static constexpr int kBytes = kTiles + (2 * STAGES + 5) * 8 + 16 + 1024;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ void mbar_arrive1(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                     ptx::smem_u32(bar))
                 : "memory");
}

// Useful tiles of the call, in raster order: experts in turn; inside an
// expert, groups of GM row tiles, column tile outer and row tile inner
// within a group, so that the CTAs at work at one time share a few weight
// tiles and a group of row tiles in L2 (each weight tile is read from DRAM
// about once per group).
struct TileMap {
    const int *first;  // [E + 1] exclusive prefix of tiles per expert (shared memory)
    int E, NT;
    const int *mtiles;  // [E] row tiles per expert (shared memory)
    int GM;             // row tiles per raster group
    __device__ void of(int t, int &e, int &mt, int &nt) const {
        const int kGroupM = GM;
        int lo = 0, hi = E - 1;  // last expert whose first tile is <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (first[mid] <= t) lo = mid; else hi = mid - 1;
        }
        e = lo;
        const int u = t - first[e], MT = mtiles[e];
        const int g = u / (kGroupM * NT);
        const int gm = min(kGroupM, MT - g * kGroupM);
        const int v = u - g * kGroupM * NT;
        nt = v / gm;
        mt = g * kGroupM + v % gm;
    }
};

// GATHER = false: the A rows of expert e are rows e * cap + j of the expert
//   planes (2-D TMA tiles), the output rows likewise.
// GATHER = true (rank planes): expert e's A rows are the receive rows
//   pair_row[pbase[e] + j], j < count[e] (pbase: exclusive prefix of the
//   counts), fetched by the loader warps; output row pbase[e] + j of the
//   pair-major output.
template <int BN, int STAGES, bool FP8, bool GATHER>
__global__ void __launch_bounds__(GATHER ? kThreadsGather : kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, const ExpertGemmParams p) {
    using L = GemmSmem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_first[kMaxExpertsExpertLayout + 1];
    __shared__ int s_mtiles[kMaxExpertsExpertLayout];
    __shared__ int s_count[kMaxExpertsExpertLayout];
    __shared__ int s_pbase[GATHER ? kMaxExpertsExpertLayout + 1 : 1];
    __shared__ volatile int s_failed;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nthreads = GATHER ? kThreadsGather : kThreads;

    const uint32_t base = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
    uint8_t *a_tiles = smem;
    uint8_t *b_tiles = smem + STAGES * L::kA;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kTiles);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;   // [2] products of a tile done
    uint64_t *acc_empty = acc_full + 2;    // [2] epilogue done with a buffer
    uint64_t *drain = acc_empty + 2;       // all products issued have finished
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    // tile list from the device-side counts
    for (int e = tid; e < p.E; e += nthreads) {
        const int c = p.recv_counts[e];
        s_count[e] = c;
        s_mtiles[e] = (c + kBM - 1) / kBM;
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // gathered rows: the B copy's arrival plus one per loader thread
            ptx::mbar_init(&full[s], GATHER ? 1 + kLoaderThreads : 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], kEpiWarps);
        }
        ptx::mbar_init(drain, 1);
        ptx::fence_mbar_init();
        s_failed = 0;
    }
    if (warp == kMmaWarp) tc::tmem_alloc(tmem_slot, 2 * BN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
        const int NT = p.N / BN;
        s_first[0] = 0;
        for (int e = 0; e < p.E; ++e) s_first[e + 1] = s_first[e] + s_mtiles[e] * NT;
        if constexpr (GATHER) {
            s_pbase[0] = 0;
            for (int e = 0; e < p.E; ++e) s_pbase[e + 1] = s_pbase[e] + s_count[e];
        }
    }
    __syncthreads();
    const uint32_t taddr = *tmem_slot;
    const TileMap tm{s_first, p.E, p.N / BN, s_mtiles, p.group_m};
    const int ntiles = s_first[p.E];
    constexpr int kBK = FP8 ? kRowBytes : kRowBytes / 2;  // values of a stage row
    const int KB = p.H / kBK;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            uint32_t kc = 0;  // k-blocks issued by this CTA, across tiles
            for (int t = blockIdx.x; t < ntiles && !s_failed; t += gridDim.x) {
                int e, mt, nt;
                tm.of(t, e, mt, nt);
                const int row0 = e * p.cap + mt * kBM, wrow0 = e * p.N + nt * BN;
                for (int kb = 0; kb < KB; ++kb, ++kc) {
                    const int s = (int)(kc % STAGES);
                    if (!ptx::mbar_wait_timed(&empty[s], ((kc / STAGES) & 1u) ^ 1u, kWaitNs)) {
                        s_failed = 1;
                        break;
                    }
                    if constexpr (GATHER) {  // A comes from the loader warps
                        ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)L::kB);
                    } else {
                        ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)(L::kA + L::kB));
                        tc::tma_load_2d(a_tiles + s * L::kA, &tmap_x, kb * kBK, row0, &full[s]);
                    }
                    tc::tma_load_2d(b_tiles + s * L::kB, &tmap_w, kb * kBK, wrow0, &full[s]);
                }
            }
            // copies still in flight land before shared memory goes away
            const uint32_t first = kc > (uint32_t)STAGES ? kc - STAGES : 0u;
            for (uint32_t k = first; k < kc; ++k)
                ptx::mbar_wait_timed(&full[k % STAGES], (k / STAGES) & 1u, kWaitNs);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc =
                FP8 ? tc::idesc_e4m3_f32(kBM, BN) : tc::idesc_bf16_f32(kBM, BN);
            uint32_t kc = 0, it = 0;
            for (int t = blockIdx.x; t < ntiles && !s_failed; t += gridDim.x, ++it) {
                const uint32_t b = it & 1u;
                if (!ptx::mbar_wait_timed(&acc_empty[b], ((it >> 1) & 1u) ^ 1u, kWaitNs)) {
                    s_failed = 1;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = taddr + b * BN;
                for (int kb = 0; kb < KB; ++kb, ++kc) {
                    const int s = (int)(kc % STAGES);
                    if (!ptx::mbar_wait_timed(&full[s], (kc / STAGES) & 1u, kWaitNs)) {
                        s_failed = 1;
                        break;
                    }
                    tc::fence_after_sync();
                    // rows written by the loaders' cp.async (generic proxy),
                    // read next by the tensor cores (async proxy)
                    if constexpr (GATHER) ptx::fence_proxy_async_smem();
                    const uint64_t ad = tc::smem_desc_sw128(ptx::smem_u32(a_tiles + s * L::kA));
                    const uint64_t bd = tc::smem_desc_sw128(ptx::smem_u32(b_tiles + s * L::kB));
                    // four K steps of 32 bytes (16 bf16 or 32 e4m3) = 2 descriptor units
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (FP8)
                            tc::mma_f8(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                        else
                            tc::mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    }
                    tc::commit(&empty[s]);  // frees the stage once these products finish
                }
                tc::commit(&acc_full[b]);  // the tile's accumulator is complete
                if (s_failed) break;
            }
            // every product issued above has finished before tensor memory is freed
            tc::commit(drain);
            ptx::mbar_wait_timed(drain, 0, kWaitNs);
        }
    } else if (GATHER && warp >= kLoaderWarp0) {
        // Loader warp w fetches tile rows 32w' .. 32w'+31 (w' = w - 6); lane l
        // knows the receive row of tile row 32w' + l.  For every k block one
        // warp instruction covers four rows: lane l copies 16-byte chunk l % 8
        // of row 4i + l / 8 (eight instructions per warp per stage, each
        // reading four whole 128-byte lines), stored at chunk position
        // c ^ (row mod 8) -- the 128-byte swizzle a TMA load would apply (the
        // stage starts on a 1024-byte boundary).  Each thread then adds one
        // arrival on the stage's barrier for when its copies have landed.
        const int lw = warp - kLoaderWarp0;
        const int c = lane & 7, sub = lane >> 3;
        const uint8_t *xb = static_cast<const uint8_t *>(p.x);
        const size_t row_bytes = (size_t)p.H * (FP8 ? 1 : 2);  // e4m3 codes or bf16
        uint32_t kc = 0;
        for (int t = blockIdx.x; t < ntiles && !s_failed; t += gridDim.x) {
            int e, mt, nt;
            tm.of(t, e, mt, nt);
            int r = mt * kBM + 32 * lw + lane;
            if (r >= s_count[e]) r = s_count[e] - 1;  // rows past the count: not stored
            long long arow = __ldg(p.pair_row + s_pbase[e] + r) & 0x7fffffff;  // (bit 31: a flag)
            if (arow >= p.a_rows) {  // guard: never produced by the pair lists
                atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                arow = 0;
            }
            // this lane's source rows for the eight instructions of a stage
            const uint8_t *src[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                src[i] = xb + (size_t)__shfl_sync(0xffffffffu, arow, 4 * i + sub) * row_bytes +
                         (c << 4);
            for (int kb = 0; kb < KB; ++kb, ++kc) {
                const int s = (int)(kc % STAGES);
                // the warp stops together (the shuffles above need whole warps)
                if (!__all_sync(0xffffffffu, ptx::mbar_wait_timed(
                                                 &empty[s], ((kc / STAGES) & 1u) ^ 1u, kWaitNs))) {
                    s_failed = 1;
                    break;
                }
                uint8_t *stage = a_tiles + s * L::kA;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = 32 * lw + 4 * i + sub;  // tile row (row mod 8 = (4i + sub) mod 8)
                    ptx::cp_async16(stage + row * kRowBytes + ((c ^ (row & 7)) << 4),
                                    src[i] + (size_t)kb * kRowBytes);
                }
                ptx::cp_async_mbar_arrive_noinc(&full[s]);
            }
        }
        ptx::cp_async_wait_all();  // copies land before shared memory goes away
    } else if (warp < kEpiWarps) {
        // epilogue: warp w owns tensor-memory lanes 32w..32w+31 = tile rows
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out);
        uint32_t it = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const uint32_t b = it & 1u;
            const bool ok = ptx::mbar_wait_timed(&acc_full[b], (it >> 1) & 1u, kWaitNs);
            __syncwarp();
            if (!ok || s_failed) {
                if (lane == 0) s_failed = 1;
                break;
            }
            tc::fence_after_sync();
            int e, mt, nt;
            tm.of(t, e, mt, nt);
            const int r = mt * kBM + 32 * warp + lane;  // row within the expert
            const bool live = r < s_count[e];
            long long orow = GATHER ? (long long)s_pbase[e] + r : (long long)e * p.cap + r;
            long long xrow = orow;  // the A row (its FP8 scale)
            // Rank planes: a row whose only local expert this is gets its
            // final message here, bf16(+0 + g * bf16(y)), in the caller's
            // output; the others' bf16 outputs go to the pair-major buffer.
            float gate = 0.0f;
            bool direct = false;
            if constexpr (GATHER) {
                xrow = 0;
                if (live) {
                    const int32_t pr = __ldg(p.pair_row + orow);
                    xrow = pr & 0x7fffffff;
                    if (xrow >= p.a_rows) xrow = 0;  // (the loaders flag such a row)
                    direct = pr < 0;  // bit 31: the row's only local expert
                    if (direct) {
                        gate = __ldg(p.pair_gate + orow);
                        orow = xrow;
                    }
                }
            }
            // FP8 operands: y = acc * sx[row] * sw[column], two fp32 products
            const float sx = (FP8 && live) ? __ldg(p.x_scale + xrow) : 1.0f;
            const float *swr = FP8 ? p.w_scale + (long long)e * p.N + (long long)nt * BN : nullptr;
            __nv_bfloat16 *dst_row =
                (direct ? reinterpret_cast<__nv_bfloat16 *>(p.final_out) : out) + orow * p.N +
                (long long)nt * BN;
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tc::ld_32x32(taddr + b * BN + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
                tc::wait_ld();
                if (FP8) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = __float_as_uint(
                            __fmul_rn(__fmul_rn(__uint_as_float(v[i]), sx), __ldg(swr + c0 + i)));
                }
                if (GATHER && direct) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float y = __bfloat162float(__float2bfloat16_rn(__uint_as_float(v[i])));
                        v[i] = __float_as_uint(__fadd_rn(0.0f, __fmul_rn(gate, y)));
                    }
                }
                if (live) {
                    uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]),
                                          __uint_as_float(v[8 * q + 1]));
                        o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]),
                                          __uint_as_float(v[8 * q + 3]));
                        o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]),
                                          __uint_as_float(v[8 * q + 5]));
                        o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]),
                                          __uint_as_float(v[8 * q + 7]));
                        dst[q] = o;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&acc_empty[b]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && s_failed) atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
    if (warp == kMmaWarp) tc::tmem_dealloc(taddr, 2 * BN);
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
bool make_map(CUtensorMap *m, const void *base, long long rows, int cols, int box_rows,
              bool fp8) {
    EncodeTiled enc = encoder();
    if (enc == nullptr) return false;
    const int esize = fp8 ? 1 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / esize), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES, bool FP8, bool GATHER>
cudaError_t launch_t(const ExpertGemmParams &p, cudaStream_t st) {
    using L = GemmSmem<BN, STAGES>;
    CUtensorMap mx, mw;
    // (gathered rows are fetched without a tensor map; mx is then unused)
    if ((!GATHER && !make_map(&mx, p.x, (long long)p.E * p.cap, p.H, kBM, FP8)) ||
        !make_map(&mw, p.w, (long long)p.E * p.N, p.H, BN, FP8))
        return cudaErrorInvalidValue;
    if (GATHER) std::memset(&mx, 0, sizeof mx);
    cudaError_t err = cudaFuncSetAttribute(expert_gemm_kernel<BN, STAGES, FP8, GATHER>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           L::kBytes);
    if (err != cudaSuccess) return err;
    // persistent: one CTA per SM (the ring fills most of shared memory), or
    // fewer when the call cannot have that many tiles
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    const long long most = (long long)p.E * p.mtiles * (p.N / BN);
    const int grid = (int)(most < sms ? most : sms);
    if (grid < 1) return cudaSuccess;
    expert_gemm_kernel<BN, STAGES, FP8, GATHER>
        <<<grid, GATHER ? kThreadsGather : kThreads, L::kBytes, st>>>(mx, mw, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gemm(const ExpertGemmParams &p, cudaStream_t st) {
    const int bk = p.fp8 ? kRowBytes : kRowBytes / 2;
    if (p.H % bk != 0 || p.H < bk || p.N % 128 != 0 || p.N < 128 || p.cap < 1 ||
        p.E > kMaxExpertsExpertLayout || p.group_m < 1)
        return cudaErrorInvalidValue;
    if (p.fp8 && (p.x_scale == nullptr || p.w_scale == nullptr)) return cudaErrorInvalidValue;
    if (p.gather) {  // rank planes: rows gathered through pair_row
        if (p.pair_row == nullptr) return cudaErrorInvalidValue;
        if (p.fp8)
            return p.N % 256 == 0 ? launch_t<256, 4, true, true>(p, st)
                                  : launch_t<128, 6, true, true>(p, st);
        return p.N % 256 == 0 ? launch_t<256, 4, false, true>(p, st)
                              : launch_t<128, 6, false, true>(p, st);
    }
    if (p.fp8)
        return p.N % 256 == 0 ? launch_t<256, 4, true, false>(p, st)
                              : launch_t<128, 6, true, false>(p, st);
    return p.N % 256 == 0 ? launch_t<256, 4, false, false>(p, st)
                          : launch_t<128, 6, false, false>(p, st);
}

}  // namespace moe
