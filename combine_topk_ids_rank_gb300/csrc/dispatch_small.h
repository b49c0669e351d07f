// dispatch_small.h -- the one-launch dispatch with FP8 receive rows
// (dispatch_small.cu) and the expert layout's one-launch dispatch
// (dispatch_small_expert.cu).  Internal to libmoe_a2a.so.
#pragma once

#include "kernels.h"

namespace moe {

// As DispatchSmallParams, in the FP8 receive format: one CTA per token
// (the whole row, so that the row's amax is one CTA reduction), its e4m3
// codes and scale stored to every destination row.
struct DispatchSmallFp8Params {
    const int32_t *topk_ids;   // [R][T][K]
    const float *topk_w;       // [R][T][K]
    const uint16_t *x;         // bf16 [R][T][H]
    uint8_t *recv_x8;          // e4m3 [R][R][m][H]
    float *recv_scale;         // [R][R][m]
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
    int R, K, E, Epr, RP, m, T, H, H8;
    unsigned long long epr_magic, T_magic;  // div_magic(Epr), div_magic(T): the launcher
};

// Threads fitted to the row (VPT 16-byte vectors each) and the row's
// shared-memory stage; dispatch_small_fp8_prepare also sets the kernels'
// shared-memory limit (once per handle).
struct DispatchSmallFp8Shape {
    int threads, vpt;
    size_t smem;
};
cudaError_t dispatch_small_fp8_prepare(int H, DispatchSmallFp8Shape *out);
cudaError_t launch_dispatch_small_fp8(const DispatchSmallFp8Params &p,
                                      const DispatchSmallFp8Shape &shape, cudaStream_t st);

// The expert layout's dispatch phase in one launch (bf16 rows, uniform T):
// the routing of route_expert.cu and the row copy, each warp deriving its
// token's rows from the ids of every token before it.  Counts are added into
// buffers that are zero on entry; the launch clears the other pair.
struct DispatchSmallExpertParams {
    const int32_t *topk_ids;   // [R][T][K]
    const float *topk_w;       // [R][T][K]
    const uint8_t *x;          // bf16 [R][T][H]
    uint8_t *recv_x;           // bf16 [E][cap][H]
    int32_t *send_row;         // [R][T][KP]
    float *wsum;               // [R][T][KP]
    int32_t *src_token;        // [E][cap]
    float *recv_w;             // [E][cap]
    int32_t *counts;           // [E] expert histogram of this call: zero on entry
    int32_t *counts_clear;     // [E] the other histogram buffer, zeroed for the next call
    int32_t *recv_counts;      // [E] rows per expert of this call: zero on entry
    int32_t *recv_counts_clear;  // [E] the other rows buffer, zeroed for the next call
    uint32_t *flags;
    uint32_t active;
    int R, K, E, Epr, KP, T, cap;
    int row_bytes, chunk_bytes, chunks, stages, stage_bytes;
    long long units;           // R * T * chunks
    unsigned long long epr_magic, chunks_magic;  // set by the launcher
};
cudaError_t dispatch_small_expert_prepare(int row_bytes, int num_sms, DispatchSmallShapes *out);
cudaError_t launch_dispatch_small_expert(const DispatchSmallExpertParams &p,
                                         const LaunchShape &shape, cudaStream_t st);

// The same with FP8 receive rows: one CTA per token (the whole row, so that
// its amax is one CTA reduction), its e4m3 codes and scale stored to each of
// its rows.  Shapes as for the rank layout's FP8 one-launch dispatch.
struct DispatchSmallExpertFp8Params {
    const int32_t *topk_ids;   // [R][T][K]
    const float *topk_w;       // [R][T][K]
    const uint16_t *x;         // bf16 [R][T][H]
    uint8_t *recv_x8;          // e4m3 [E][cap][H]
    float *recv_scale;         // [E][cap]
    int32_t *send_row;         // [R][T][KP]
    float *wsum;               // [R][T][KP]
    int32_t *src_token;        // [E][cap]
    float *recv_w;             // [E][cap]
    int32_t *counts, *counts_clear, *recv_counts, *recv_counts_clear;  // as above
    uint32_t *flags;
    uint32_t active;
    int R, K, E, Epr, KP, T, cap, H, H8;
    unsigned long long epr_magic;  // set by the launcher
};
cudaError_t dispatch_small_expert_fp8_prepare(int H, DispatchSmallFp8Shape *out);
cudaError_t launch_dispatch_small_expert_fp8(const DispatchSmallExpertFp8Params &p,
                                             const DispatchSmallFp8Shape &shape, cudaStream_t st);

}  // namespace moe
