// expert.h -- parameter blocks and host launchers of the expert-side
// products (expert_gemm.cu, expert_rank.cu).  Internal to libmoe_a2a.so.
#pragma once

#include "kernels.h"

namespace moe {

// Expert-side grouped product over the expert planes (expert_gemm.cu).
struct ExpertGemmParams {
    const void *x;               // bf16 [E][cap][H]
    const void *w;               // bf16 [E][N][H]
    void *out;                   // bf16 [E][cap][N]
    const int32_t *recv_counts;  // [E]
    const float *x_scale;        // FP8 operands: [E][cap] row scales, else null
    const float *w_scale;        // FP8 operands: [E][N] channel scales, else null
    uint32_t *flags;
    int E, cap, H, N, mtiles;    // mtiles = ceil(cap / 128) (an upper bound of row tiles)
    int fp8;                     // 1: x and w are e4m3 codes (x_scale, w_scale used)
    // Rank planes (gather = 1): x is the bf16 receive region [rows][H];
    // recv_counts holds the pair count of each expert, pair_row the receive
    // row of each pair (expert-major, pbase[e] = prefix of the counts) and
    // out is pair-major [pairs][N].
    int gather;
    const int32_t *pair_row;     // [pairs]: receive row; bit 31 set when it is the row's
                                 // only local expert (its message is written here)
    const float *pair_gate;      // [pairs]: the gate of such a row's expert
    void *final_out;             // bf16 [rows][N]: messages of single-expert rows
    long long a_rows;            // rows of x (gather guard)
    int group_m;                 // row tiles per raster group
};
cudaError_t launch_expert_gemm(const ExpertGemmParams &p, cudaStream_t st);

// Rank planes: pair lists and the gated per-row sum of the experts' outputs
// (expert_rank.cu).
struct RankPairsParams {
    const int32_t *recv_ids;     // [R][R][m][K]: local expert or -1
    const float *recv_w;         // [R][R][m][K]
    const int32_t *recv_counts;  // [R][R]
    const int32_t *pair_counts;  // [E]: local_expert_counts of the dispatch
    int32_t *cursor;             // [E + 1], zero on entry: pairs placed per expert, then
                                 // the number of rows with several local experts
    int32_t *pair_row;           // [pairs]: receive row of each pair, expert-major; bit
                                 // 31 set when it is the row's only local expert
    float *pair_gate;            // [pairs]: the gate of such a row's expert
    int32_t *pair_of;            // [R][R][m][K]: pair of (row, k), -1 if none
    int32_t *multi;              // [multi_cap]: the rows with several local experts
                                 // (in no particular order; count in cursor[E])
    long long multi_cap;
    const uint16_t *y;           // [pairs][N] bf16 expert outputs
    uint16_t *out;               // [R][R][m][N] bf16 messages
    uint32_t *flags;             // device flag word (consistency guard)
    int R, m, K, E, N;
    int apply_gates;
};
cudaError_t launch_rank_pairs(const RankPairsParams &p, int num_sms, cudaStream_t st);
cudaError_t launch_rank_aggregate(const RankPairsParams &p, int num_sms, cudaStream_t st);

}  // namespace moe
