// kernels.h -- parameter blocks and host launchers of the kernels of the
// dispatch / combine path (the expert-side products: expert.h).  Internal
// to libmoe_a2a.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace moe {

constexpr int kMaxRanks = 32;

// The tokens of one call: source rank s holds count[s] tokens, stored at rows
// s * stride + t (t < count[s]) of the [R][stride] token arrays; first[s] is
// the exclusive prefix of the counts (first[R] = all tokens).  The uniform
// case is count[s] = stride = T.
struct TokenMap {
    int stride;
    int uniform;  // every count equals stride
    int count[kMaxRanks];
    int first[kMaxRanks + 1];
};

// (source, token) of the i-th token of the call, i < first[R].
__host__ __device__ inline void token_of(const TokenMap &m, int R, long long i, int &s,
                                         int &t) {
    if (m.uniform) {
        // i < R * stride <= 2^29: a 32-bit division suffices
        s = (int)((uint32_t)i / (uint32_t)m.stride);
    } else {
        s = 0;
        while (s + 1 < R && i >= m.first[s + 1]) ++s;
    }
    t = (int)(i - m.first[s]);
}

// Division by a divisor D fixed for a launch, as a multiply-high: with
// magic = ceil(2^32 / D), floor(n * magic / 2^32) = floor(n / D) for every
// n >= 0 with n * D < 2^32.  Used where both stay below 2^16: the owner rank
// of an expert, e / Epr (ids and Epr below 2^13, MOE_MAX_EXPERTS), and the
// small dispatch's unit / chunks and token / T.  The launchers fill the
// magics themselves.
inline unsigned long long div_magic(int D) {
    return ((1ull << 32) + (unsigned long long)D - 1) / (unsigned long long)D;
}
inline unsigned long long owner_magic(int Epr) { return div_magic(Epr); }
#ifdef __CUDACC__
__device__ __forceinline__ int div_by(int n, unsigned long long magic) {
    return (int)(((unsigned long long)(unsigned)n * magic) >> 32);
}
__device__ __forceinline__ int owner_of(int e, unsigned long long magic) {
    return div_by(e, magic);
}
#endif

// Largest number of tokens per CTA of the two routing kernels (one token
// per thread); the tile of a call is 32, 64, 128 or 256.
constexpr int kRouteTile = 256;
constexpr int kRouteMinTile = 32;

// Tuning switches, for sweeps only: read from the environment once, when a
// handle is created (read_tuning in moe_a2a.cpp), never on the call path.
// 0 selects the measured default of each.
struct Tuning {
    int route_overlap;         // MOE_ROUTE_OVERLAP: 0 = passes in stream order (default 1)
    int route_tile;            // MOE_ROUTE_TILE: 32, 64, 128 or 256 tokens
    int dispatch_stages;       // MOE_DISPATCH_STAGES: ring depth of the bf16 row copy
    int dispatch_ctas_per_sm;  // MOE_DISPATCH_CTAS_PER_SM
    int fp8_dispatch_stages;   // MOE_FP8_DISPATCH_STAGES: 2..8
    int combine_kernel;        // MOE_COMBINE_KERNEL: 1 = ring, 2 = registers
    int combine_ring_slots;    // MOE_COMBINE_RING_SLOTS: 2..32
    int dispatch_small_max;    // MOE_DISPATCH_SMALL_MAX: largest T for the one-launch
                               // dispatch (0: the default, -1: never)
    int gemm_group_m;          // MOE_GEMM_GROUP_M: row tiles per raster group of the
                               // expert product
    int combine_small_max;     // MOE_COMBINE_SMALL_MAX: most tokens (all sources) for the
                               // cluster combine (0: the default, -1: never)
};

// Tile of one call: 256 tokens.  Smaller tiles (more CTAs per SM) measured
// slower on every shape tried -- wide EP 206.6 us at 32 vs 199-200 us at
// 128-256, prefill 321.5 vs 318.8, decode 32.0 vs 31.4 (dispatch phase) --
// since the work per token is a few dependent memory accesses and more CTAs
// only add scan steps.  Tuning::route_tile overrides.
inline int route_tile(const Tuning &tn) {
    const int t = tn.route_tile;
    return (t == 32 || t == 64 || t == 128 || t == 256) ? t : kRouteTile;
}

// Routing, pass 1: per-tile destination counts, their exclusive per-tile
// prefixes (by the last tile of each source), recv counts, the expert
// histogram accumulated with atomics.
struct RouteCountParams {
    const int32_t *topk_ids;  // [R][T][K]
    int32_t *tile_counts;     // [R][ntiles][RP]
    int32_t *tile_prefix;     // [R][ntiles][RP]
    int32_t *tile_ticket;     // [R], zero between calls
    int32_t *hist_accum;      // [R][E], zero between calls
    int32_t *recv_counts;     // [R][R]
    int32_t *local_slot;      // [R][T][RP] slots inside the token's tile, or null
    uint32_t *flags;          // sticky device flag word
    TokenMap map;
    uint32_t active;          // ranks that receive messages
    int R, K, E, Epr, RP, ntiles, tile;
    unsigned long long epr_magic;  // owner_magic(Epr), set by the launcher
};

// Routing, pass 2: slots (ascending token order per plane), send table,
// per-destination weights, source map, masked metadata rows, counts.
struct RouteScanParams {
    const int32_t *topk_ids;   // [R][T][K]
    const float *topk_w;       // [R][T][K]
    const int32_t *tile_prefix;
    int32_t *hist_accum;       // read, then set back to zero
    int32_t *send_slot;        // [R][T][RP]
    float *dest_weight;        // [R][T][RP]
    int32_t *src_token;        // [R][R][m]
    int32_t *recv_ids;         // [R][R][m][K]
    float *recv_w;             // [R][R][m][K]
    int8_t *topk_dest;         // [R][T][K] or null: rank whose message slot k carries
    int32_t *local_counts;     // [E]  (= [R][Epr])
    TokenMap map;
    uint32_t active;
    int R, K, E, Epr, RP, m, ntiles, tile;
    int dg;                    // destinations per CTA (1 or 4): grid z = RP / dg
    unsigned long long epr_magic;  // owner_magic(Epr), set by the launcher
};

// Expert-major layout routing (route_expert.cu).
constexpr int kMaxTopK = 32;
constexpr int kMaxExpertsExpertLayout = 1024;
struct RouteExpertParams {
    const int32_t *topk_ids;  // [R][stride][K]
    const float *topk_w;      // [R][stride][K]
    int32_t *tile_counts;     // [R][ntiles][E]
    int32_t *send_row;        // [R][stride][KP]: absolute row of the expert planes or -1
    float *wsum;              // [R][stride][KP]
    int32_t *src_token;       // [E][cap]: s * stride + t
    float *recv_w;            // [E][cap]
    int32_t *recv_counts;     // [E]
    int32_t *hist_accum;      // [E], zero between calls: pass 1 adds, pass 2 moves it out
    int32_t *local_counts;    // [E], written by pass 2
    uint32_t *flags;
    TokenMap map;
    uint32_t active;
    int R, K, E, Epr, KP, cap, ntiles;
    int kg;                   // top-k slots per CTA of the second pass: grid z = KP / kg
};
int route_expert_tile();
cudaError_t launch_route_expert(const RouteExpertParams &p, cudaStream_t st);

// Where the entries of a token's send row point.  Rank layout: entry d is
// the token's slot in plane (d, s), i.e. row (d * R + s) * m + slot of the
// receive region.  Expert layout: entry k already is the absolute row
// (e * cap + slot) of the expert planes.
struct DestRows {
    int P;           // entries per send row: RP (rank) or KP (expert)
    int expert;      // 0: rank planes, 1: absolute rows
    long long rows;  // rows of the receive region (expert layout guard)
    int cap;         // rows per expert plane (expert layout)
    int Epr;         // experts per rank (expert layout: owner of a row)
};

// Row of the receive region for send-row entry d holding v >= 0, or -1 if
// v lies outside its plane (a guard; never produced by the routing pass).
__device__ __forceinline__ long long dest_row(const DestRows &D, int R, int m, int d, int s,
                                              int v) {
    if (D.expert) return v < D.rows ? (long long)v : -1;
    return v < m ? ((long long)d * R + s) * m + v : -1;
}

// The same row for an entry already checked with dest_row (no guard, no
// branch: for the load-issue paths of the combines).
__device__ __forceinline__ long long dest_row_checked(const DestRows &D, int R, int m, int d,
                                                      int s, int v) {
    return D.expert ? (long long)v : ((long long)d * R + s) * m + v;
}

// Rank that owns send-row entry d holding v >= 0 (for the active-rank test).
__device__ __forceinline__ int dest_rank(const DestRows &D, int d, int v) {
    return D.expert ? (v / D.cap) / D.Epr : d;
}

// Dispatch rows: x[s][t] -> recv_x[d][s][slot] for every destination of
// the token, staged through shared memory with bulk asynchronous copies.
struct DispatchParams {
    const uint8_t *x;          // bf16 [R][T][H] as bytes
    const int32_t *send_slot;  // [R][T][RP]
    uint8_t *recv_x;           // bf16 receive rows as bytes
    uint32_t *flags;
    TokenMap map;
    DestRows dest;
    // Rank layout straight after route_count: send_slot holds slots inside
    // the token's tile and tile_prefix the tiles' exclusive prefixes; else
    // (tile_prefix null) send_slot holds the final entries.
    const int32_t *tile_prefix;  // [R][ntiles][RP] or null
    int tile, ntiles;
    int R, RP, m;
    int row_bytes;             // 2H
    int chunk_bytes;           // <= row_bytes, multiple of 16
    int chunks;                // ceil(row_bytes / chunk_bytes)
    int stages;                // shared-memory ring depth
    int stage_bytes;           // chunk_bytes + meta, 128-byte multiple
    long long units;           // tokens * chunks
};

// Combine: ascending-rank fp32 gather-sum of each token's messages, with
// the optional fused residual add + RMSNorm epilogue.
struct CombineParams {
    const uint16_t *expert_out;   // bf16 [R][R][m][H]
    const int32_t *send_slot;     // [R][T][RP]
    const float *dest_weight;     // [R][T][RP]
    const uint16_t *residual;     // bf16 [R][T][H] or null
    const uint16_t *gamma;        // bf16 [H] or null
    uint16_t *out;                // bf16 [R][T][H]
    uint16_t *residual_out;       // bf16 [R][T][H] or null
    uint8_t *out8;                // e4m3 [R][T][H] (FP8 output variant) or null
    float *out_scale;             // [R][T] (FP8 output variant) or null
    uint32_t *flags;
    float eps;
    TokenMap map;
    DestRows dest;
    uint32_t active;              // ranks whose messages are summed
    int R, RP, m, H, H8;          // H8 = H / 8 (16-byte vectors per row)
    int ring_slots;               // shared-memory row buffers (ring kernel)
    long long tokens;             // map.first[R]
};

// Combine for small batches (combine_small.cu): each token's row split over
// a cluster of kClusterCtas CTAs; bf16 output.
constexpr int kClusterCtas = 4;
constexpr int kSmallCombineMaxThreads = 256;
struct SmallCombineShape {
    int cluster;  // CTAs per token
    int cols8;    // 16-byte vectors of the row per CTA
    int vpt;      // vectors per thread (1 or 2)
    int threads;  // per CTA
};
bool combine_small_shape(int H, SmallCombineShape *sh);
cudaError_t launch_combine_small(const CombineParams &p, bool weighted, bool fused,
                                 const SmallCombineShape &sh, cudaStream_t st);

// Compatibility combine: bf16 pairwise tree over the top-k slots.
struct CombineTreeParams {
    const uint16_t *expert_out;  // bf16 [R][R][m][H]
    const int32_t *send_slot;    // [R][T][RP]
    const int8_t *topk_dest;     // [R][T][K]
    const uint16_t *residual;    // bf16 [R][T][H] or null
    const uint16_t *gamma;       // bf16 [H] or null
    uint16_t *out;
    uint16_t *residual_out;
    uint32_t *flags;
    float eps;
    TokenMap map;
    uint32_t active;
    int R, RP, m, H, H8, K, P;  // P = K rounded up to a power of two (<= 8)
    long long tokens;
};

struct LaunchShape {
    int grid;
    int block;
    size_t smem;
};

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel of the stream finishes.  Only for
// kernels that run griddepcontrol.wait before touching anything an earlier
// kernel writes or reads.
template <typename Kern, typename... Args>
inline cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_route_count(const RouteCountParams &p, cudaStream_t st);
cudaError_t launch_route_scan(const RouteScanParams &p, cudaStream_t st, bool pdl);

// Dispatch: ring depth and per-SM residency for a row size and P send-row
// entries per token.
cudaError_t dispatch_prepare(int row_bytes, int P, int num_sms, const Tuning &tn,
                             DispatchParams *p, LaunchShape *shape);
cudaError_t launch_dispatch_rows(const DispatchParams &p, const LaunchShape &shape,
                                 cudaStream_t st, bool pdl);

// Combine: vectors per thread, block size and grid for a hidden size.
cudaError_t combine_prepare(int H, bool weighted, bool fused, int num_sms,
                            LaunchShape *shape, int *vpt);
cudaError_t launch_combine(const CombineParams &p, bool weighted, bool fused, int vpt,
                           const LaunchShape &shape, cudaStream_t st);

// Combine with bulk-copy row streaming (one CTA per SM, producer warp +
// consumer warps): vectors per consumer thread, ring depth and shape.
cudaError_t combine_ring_prepare(int H, bool weighted, bool fused, bool out8, int num_sms,
                                 const Tuning &tn, LaunchShape *shape, int *vpt, int *slots);
cudaError_t launch_combine_ring(const CombineParams &p, bool weighted, bool fused, bool out8,
                                int vpt, const LaunchShape &shape, cudaStream_t st);

// The whole dispatch phase in one launch for batches of at most one routing
// tile per source (dispatch_small.cu; rank layout, bf16 rows, uniform T).
constexpr int kSmallMaxChunks = 8;
struct DispatchSmallParams {
    const int32_t *topk_ids;   // [R][T][K]
    const float *topk_w;       // [R][T][K]
    const uint8_t *x;          // bf16 [R][T][H] as bytes
    uint8_t *recv_x;           // bf16 [R][R][m][H] as bytes
    int32_t *send_slot;        // [R][T][RP]
    float *dest_weight;        // [R][T][RP]
    int32_t *src_token;        // [R][R][m]
    int32_t *recv_ids;         // [R][R][m][K]
    float *recv_w;             // [R][R][m][K]
    int8_t *topk_dest;         // [R][T][K] or null
    int32_t *recv_counts;      // [R][R]
    int32_t *counts;           // [E] local-expert counts of this call: zero on entry
    int32_t *counts_clear;     // [E] the other counts buffer, zeroed for the next call
    uint32_t *flags;
    uint32_t active;
    int R, K, E, Epr, RP, m, T;
    int row_bytes, chunk_bytes, chunks, stages, stage_bytes;
    long long units;           // R * T * chunks
    unsigned long long epr_magic;  // owner_magic(Epr), set by the launcher
    unsigned long long chunks_magic, T_magic;  // div_magic(chunks), div_magic(T): launcher
};
struct DispatchSmallShapes {   // per chunk count 1..kSmallMaxChunks
    int chunk_bytes[kSmallMaxChunks + 1], chunks[kSmallMaxChunks + 1];
    int stage_bytes[kSmallMaxChunks + 1];
    LaunchShape shape[kSmallMaxChunks + 1];
    int stages;
};
cudaError_t dispatch_small_prepare(int row_bytes, int num_sms, DispatchSmallShapes *out);
int dispatch_small_chunks(int row_bytes, int num_sms, long long tokens);
cudaError_t launch_dispatch_small(const DispatchSmallParams &p, const LaunchShape &shape,
                                  cudaStream_t st);

// Dispatch with FP8 rows: per-token e4m3 quantisation into the receive
// planes plus a per-row scale (see dispatch_fp8.cu).
struct DispatchFp8Params {
    const uint16_t *x;        // bf16 [R][T][H]
    const int32_t *send_slot; // [R][T][RP]; tile-local slots when tile_prefix is set
    const int32_t *tile_prefix;  // [R][ntiles][RP] or null
    int tile, ntiles;
    uint8_t *recv_x8;         // e4m3 receive rows [rows][H]
    float *recv_scale;        // [rows]
    uint32_t *flags;
    TokenMap map;
    DestRows dest;
    int R, RP, m, H, H8;
    int stages;               // set by dispatch_fp8_prepare
    long long tokens;
};
// Ring depth, residency and function attributes of the FP8 dispatch for a
// hidden size (once per handle): fills p->stages and the launch shape.
cudaError_t dispatch_fp8_prepare(int H, int num_sms, const Tuning &tn, DispatchFp8Params *p,
                                 LaunchShape *shape);
cudaError_t launch_dispatch_fp8(const DispatchFp8Params &p, const LaunchShape &shape,
                                cudaStream_t st);
// fp32 rows [rows][H] -> e4m3 codes [rows][H] + scale [rows] (H % 8 == 0).
cudaError_t launch_quantize_rows_fp8(const float *x, long long rows, int H, uint8_t *q,
                                     float *scale, int num_sms, cudaStream_t st);

cudaError_t launch_combine_tree(const CombineTreeParams &p, int num_sms, cudaStream_t st);

}  // namespace moe
