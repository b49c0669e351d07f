/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the top-k
 * expert-parallel dispatch / combine path on logical ranks.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load it (through oracle/oracle.py).  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Every function below is the plain definition written as nested loops, in
 * the order the definition states it.  Build flags: -O2 -ffp-contract=off,
 * no -ffast-math, so every float operation is one IEEE-754 binary32
 * round-to-nearest-even operation and no multiply-add is ever contracted.
 *
 * Sources (web pages; cited by title and section):
 *   [IX]  SemiAnalysisAI/InferenceX PR #2450, "CollectiveX: add FlashInfer
 *         one-sided NVLink EP for the GB SKUs" -- "The adapter" table
 *         (phase contract, padded receive [ep_size, runtime_max, hidden],
 *         workspace sized once), the bring-up "run" table (routing metadata
 *         as payloads 2/3, non-local expert-id masking, local_expert_counts),
 *         "Kernel arithmetic read from source" (fp32 accumulate, one
 *         round-to-nearest-even narrowing), "Synthesis" table (dedup: a
 *         duplicate-rank message is read once; partial routing compacts),
 *         "Update -- the correctness failures are resolved" ("domain-fp32":
 *         fp32 accumulator, single narrowing store).
 *   [VL]  vllm-project/vllm PR #41382, "[Bugfix] Fix double reduce in
 *         flashinfer_nvlink_two_sided and flashinfer_nvlink_one_sided
 *         backends" -- the combine output is already reduced; it is final.
 *   [MG]  magik.net, "Fusing the Allreduce: A Precision Investigation into
 *         FlashInfer's Verify-Path Optimization" -- "The Message Itself":
 *         reduce(h) followed by residual-add + RMSNorm, done as one step.
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes of the repository):
 *   - expert e lives on rank owner(e) = e / (E / R)  (contiguous placement);
 *   - slot order inside a (destination, source) plane is ascending source
 *     token index;
 *   - the per-destination weight wd(s,t,d) is the fp32 sum, in ascending k,
 *     of the top-k weights whose expert lives on d, starting from +0.0f;
 *   - the combine sums messages over destinations in ascending rank order,
 *     starting from +0.0f, in fp32, and narrows once;
 *   - expert id -1 means "no expert" and is skipped; any other id outside
 *     [0, E) is counted as invalid and also skipped;
 *   - fused epilogue: hsum = acc + residual (fp32), residual_out =
 *     bf16(hsum), y = hsum / sqrt(mean(hsum^2) + eps) * gamma, the mean of
 *     squares and the square root taken in double here (the accuracy
 *     reference), y narrowed to bf16 once.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32, from the IEEE-754 definition                       */
/* ------------------------------------------------------------------------ */

/* A bfloat16 is the upper 16 bits of a binary32.  Widening is exact. */
float oracle_f32_from_bf16(uint16_t b)
{
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Narrowing with round-to-nearest, ties-to-even.  The 16 dropped bits are
 * compared with one half of the kept unit in the last place: above half
 * rounds up, below half rounds down, exactly half rounds to the even kept
 * value.  A carry out of the mantissa bumps the exponent (and turns the
 * largest finite values into infinity), as IEEE rounding requires.  NaN stays
 * NaN (made quiet so that dropping payload bits cannot turn it into inf). */
uint16_t oracle_bf16_from_f32(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint32_t exponent = (bits >> 23) & 0xffu;
    uint32_t mantissa = bits & 0x7fffffu;
    if (exponent == 0xffu && mantissa != 0u)
        return (uint16_t)((bits >> 16) | 0x0040u);
    uint32_t kept = bits >> 16;
    uint32_t dropped = bits & 0xffffu;
    const uint32_t half = 0x8000u;
    if (dropped > half || (dropped == half && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------------ */
/* a1: routing, per-destination dedup, slot assignment, counts               */
/* ------------------------------------------------------------------------ */

/*
 * Inputs
 *   topk_ids [R][T][K] int32, topk_w [R][T][K] float: source rank s holds T
 *   tokens, each with K expert ids and K weights.
 * Outputs (all written in full)
 *   dmask     [R][T]     bit d set iff token (s,t) has a valid expert on d
 *   wd        [R][T][R]  per-destination weight (0.0f where not sent)
 *   send_slot [R][T][R]  slot of (s,t) in plane (d,s), -1 where not sent
 *   recv_counts [R][R]   [d][s]: rows of source s received by d
 *   src_token [R][R][m]  [d][s][j]: the source token in slot j, -1 past count
 *   local_expert_counts [R][E/R]: valid (token, k) entries per local expert
 * Returns the number of invalid ids (outside [-1, E)), which are skipped.
 *
 * [IX] "Synthesis": a token reaches each distinct destination rank once, so
 * duplicate experts on one rank are read once; partial routing compacts each
 * plane.  [IX] run table: recv counters are the authoritative per-source
 * counts.  Placement and slot order are the readings listed at the top.
 */
long oracle_route(int R, int T, int K, int E, int m,
                  const int32_t *topk_ids, const float *topk_w,
                  uint32_t *dmask, float *wd, int32_t *send_slot,
                  int32_t *recv_counts, int32_t *src_token,
                  int32_t *local_expert_counts)
{
    const int Epr = E / R;
    long invalid = 0;

    for (int i = 0; i < R * (E / R); ++i)
        local_expert_counts[i] = 0;

    /* Destination set and per-destination weight of every token. */
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < T; ++t) {
            const int32_t *ids = topk_ids + ((size_t)s * T + t) * K;
            const float *w = topk_w + ((size_t)s * T + t) * K;
            uint32_t mask = 0u;
            for (int k = 0; k < K; ++k) {
                int32_t e = ids[k];
                if (e == -1)
                    continue;
                if (e < -1 || e >= E) {
                    invalid += 1;
                    continue;
                }
                int d = e / Epr;
                mask |= 1u << d;
                local_expert_counts[d * Epr + (e - d * Epr)] += 1;
            }
            dmask[(size_t)s * T + t] = mask;

            for (int d = 0; d < R; ++d) {
                float sum = 0.0f;
                for (int k = 0; k < K; ++k) {
                    int32_t e = ids[k];
                    if (e < 0 || e >= E)
                        continue;
                    if (e / Epr == d)
                        sum = sum + w[k];
                }
                wd[((size_t)s * T + t) * R + d] = sum;
            }
        }
    }

    /* Slots: in plane (d, s) the tokens that go to d, in ascending t. */
    for (size_t i = 0; i < (size_t)R * R * m; ++i)
        src_token[i] = -1;
    for (int s = 0; s < R; ++s) {
        for (int d = 0; d < R; ++d) {
            int32_t count = 0;
            for (int t = 0; t < T; ++t) {
                size_t at = ((size_t)s * T + t) * R + d;
                if (dmask[(size_t)s * T + t] & (1u << d)) {
                    send_slot[at] = count;
                    src_token[((size_t)d * R + s) * m + count] = t;
                    count += 1;
                } else {
                    send_slot[at] = -1;
                }
            }
            recv_counts[d * R + s] = count;
        }
    }
    return invalid;
}

/* ------------------------------------------------------------------------ */
/* a2: dispatch -- copy rows and routing metadata into the padded planes     */
/* ------------------------------------------------------------------------ */

/*
 * recv_x   [R][R][m][H] bf16:  recv_x[d][s][j] = x[s][src_token[d][s][j]]
 * recv_ids [R][R][m][K] int32: the token's expert id where it lives on d,
 *                              -1 elsewhere (non-local masking)
 * recv_w   [R][R][m][K] float: the token's weight where local, 0.0f elsewhere
 * Only slots j < recv_counts[d][s] are written; padding is left as it was.
 *
 * [IX] "The adapter": receive is padded [ep_size, runtime_max, hidden], only
 * valid slots are meaningful.  [IX] run table: routing metadata travels as
 * payloads 2/3 and non-local expert ids are masked to -1.
 */
void oracle_dispatch(int R, int T, int K, int E, int H, int m,
                     const int32_t *topk_ids, const float *topk_w,
                     const uint16_t *x, const int32_t *recv_counts,
                     const int32_t *src_token, uint16_t *recv_x,
                     int32_t *recv_ids, float *recv_w)
{
    const int Epr = E / R;
    for (int d = 0; d < R; ++d) {
        for (int s = 0; s < R; ++s) {
            int32_t count = recv_counts[d * R + s];
            for (int j = 0; j < count; ++j) {
                size_t slot = ((size_t)d * R + s) * m + j;
                int t = src_token[slot];
                const uint16_t *row = x + ((size_t)s * T + t) * H;
                for (int h = 0; h < H; ++h)
                    recv_x[slot * H + h] = row[h];
                for (int k = 0; k < K; ++k) {
                    int32_t e = topk_ids[((size_t)s * T + t) * K + k];
                    int local = (e >= 0 && e < E && e / Epr == d);
                    recv_ids[slot * K + k] = local ? e : -1;
                    recv_w[slot * K + k] = local ? topk_w[((size_t)s * T + t) * K + k] : 0.0f;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* a4: the fused epilogue of one reduced row (shared by every combine)       */
/* ------------------------------------------------------------------------ */

/*
 * acc[0..H): the token's reduced fp32 row.  res_row == NULL: unfused,
 * out_row = bf16(acc), y_row = acc.  Otherwise hsum = acc + f32(res_row)
 * (fp32 add), rout_row = bf16(hsum) (if not NULL), ms = sum hsum^2 / H
 * (double), y = hsum * (1 / sqrt(ms + eps)) * f32(gamma) (double), y_row = y,
 * out_row = bf16((float)y).  hsum is scratch of H floats.
 * [MG] "The Message Itself": residual add + RMSNorm after the reduction.
 */
static void finish_row(int H, const float *acc, const uint16_t *res_row,
                       const uint16_t *gamma, float eps, float *hsum,
                       uint16_t *out_row, uint16_t *rout_row, double *y_row)
{
    if (res_row == 0) {
        /* unfused: the reduced sum is the output, narrowed once */
        for (int h = 0; h < H; ++h) {
            out_row[h] = oracle_bf16_from_f32(acc[h]);
            if (y_row)
                y_row[h] = (double)acc[h];
        }
        return;
    }
    /* residual add, then RMSNorm of the fp32 sum */
    double sumsq = 0.0;
    for (int h = 0; h < H; ++h) {
        hsum[h] = acc[h] + oracle_f32_from_bf16(res_row[h]);
        if (rout_row)
            rout_row[h] = oracle_bf16_from_f32(hsum[h]);
        sumsq += (double)hsum[h] * (double)hsum[h];
    }
    double inv = 1.0 / sqrt(sumsq / (double)H + (double)eps);
    for (int h = 0; h < H; ++h) {
        double y = (double)hsum[h] * inv * (double)oracle_f32_from_bf16(gamma[h]);
        if (y_row)
            y_row[h] = y;
        out_row[h] = oracle_bf16_from_f32((float)y);
    }
}

/* ------------------------------------------------------------------------ */
/* a3 + a4: combine (reduce once, ascending rank, fp32) and fused epilogue   */
/* ------------------------------------------------------------------------ */

/*
 * For each requested token (flat index s*T + t; tokens == NULL means all
 * R*T tokens in order), writing row i of every output for the i-th token:
 *
 *   acc[h] = sum over destinations d in dmask(s,t), ascending d, of
 *            v = f32(expert_out[d][s][send_slot(s,t,d)][h])        (weighted=0)
 *            wd(s,t,d) * v                                        (weighted=1)
 *            starting from +0.0f, one fp32 multiply and one fp32 add each.
 *   acc_out[i][h] = acc[h]                                        (if not NULL)
 *
 * Unfused (residual == NULL): out[i][h] = bf16(acc[h]); y_ref = acc.
 * Fused: hsum = acc + f32(residual[s][t][h])            (fp32 add)
 *        residual_out[i][h] = bf16(hsum)
 *        ms  = sum_h hsum^2 / H                          (double)
 *        y   = hsum * (1 / sqrt(ms + eps)) * f32(gamma[h])  (double)
 *        y_ref[i][h] = y, out[i][h] = bf16((float)y)
 *
 * [IX] "Kernel arithmetic read from source" and "Update": fp32 accumulation
 * with one round-to-nearest-even narrowing.  [VL]: the result is reduced
 * exactly once.  [MG] "The Message Itself": residual add + RMSNorm after the
 * reduction.
 */
void oracle_combine(int R, int T, int H, int m, int weighted,
                    const uint32_t *dmask, const int32_t *send_slot,
                    const float *wd, const uint16_t *expert_out,
                    const uint16_t *residual, const uint16_t *gamma, float eps,
                    const int64_t *tokens, long ntokens,
                    float *acc_out, uint16_t *out, uint16_t *residual_out,
                    double *y_ref)
{
    long n = tokens ? ntokens : (long)R * T;
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    float *hsum = (float *)malloc((size_t)H * sizeof(float));
    if (!acc || !hsum) {
        free(acc);
        free(hsum);
        return;
    }
    for (long i = 0; i < n; ++i) {
        long flat = tokens ? (long)tokens[i] : i;
        int s = (int)(flat / T);
        int t = (int)(flat % T);
        uint32_t mask = dmask[flat];
        size_t o = (size_t)i * H;

        /* a3: one message per destination rank, ascending rank, fp32 */
        for (int h = 0; h < H; ++h) {
            float a = 0.0f;
            for (int d = 0; d < R; ++d) {
                if (!(mask & (1u << d)))
                    continue;
                int32_t j = send_slot[(size_t)flat * R + d];
                size_t row = ((size_t)d * R + s) * m + (size_t)j;
                float v = oracle_f32_from_bf16(expert_out[row * H + h]);
                if (weighted) {
                    float p = wd[(size_t)flat * R + d] * v;
                    a = a + p;
                } else {
                    a = a + v;
                }
            }
            acc[h] = a;
            if (acc_out)
                acc_out[o + h] = a;
        }

        finish_row(H, acc, residual ? residual + ((size_t)s * T + t) * H : 0, gamma, eps,
                   hsum, out + o, residual_out ? residual_out + o : 0, y_ref ? y_ref + o : 0);
    }
    free(acc);
    free(hsum);
}

/* ------------------------------------------------------------------------ */
/* Compatibility reduction: bf16 pairwise tree over the top-k slots          */
/* ------------------------------------------------------------------------ */

/*
 * [IX] "Update -- the correctness failures are resolved": through version
 * 0.6.15 FlashInfer's one-sided combine keeps one accumulator per top-k
 * slot in the payload type (bf16), with each operand at its original top-k
 * slot (duplicate-rank slots are blanked in place, not compacted), and
 * reduces the slots with a pairwise tree -- (a0+a1)(a2+a3)(a4+a5)(a6+a7),
 * then (a0+a2)(a4+a6), then (a0+a4) -- rounding to bf16 after every add.
 *
 * For each requested token (flat s*T + t; tokens == NULL means all):
 *   slot k holds f32(expert_out[d][s][send_slot(s,t,d)][h]) when e_k is a
 *   valid expert, d = owner(e_k), and no earlier slot k' < k has a valid
 *   expert on the same rank d; otherwise slot k holds 0.
 *   The K slots are padded with zeros to the next power of two P; for
 *   stride = 1, 2, 4, ... < P: a[i] = bf16(a[i] + a[i + stride]) for every i
 *   that is a multiple of 2*stride.  The result is a[0] (already bf16).
 * Unfused (residual == NULL): out = a[0].  Fused: the same epilogue as
 * oracle_combine with acc = a[0]: hsum = acc + residual (fp32),
 * residual_out = bf16(hsum), y = hsum / sqrt(mean(hsum^2) + eps) * gamma.
 * The reduction is unweighted, as FlashInfer's combine is.
 */
void oracle_combine_topk_tree(int R, int T, int K, int E, int H, int m,
                              const int32_t *topk_ids, const int32_t *send_slot,
                              const uint16_t *expert_out, const uint16_t *residual,
                              const uint16_t *gamma, float eps,
                              const int64_t *tokens, long ntokens,
                              uint16_t *out, uint16_t *residual_out, double *y_ref)
{
    const int Epr = E / R;
    int P = 1;
    while (P < K)
        P *= 2;
    long n = tokens ? ntokens : (long)R * T;
    int *slot_dest = (int *)malloc((size_t)P * sizeof(int));
    float *a = (float *)malloc((size_t)P * sizeof(float));
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    float *hsum = (float *)malloc((size_t)H * sizeof(float));
    if (!slot_dest || !a || !acc || !hsum) {
        free(slot_dest);
        free(a);
        free(acc);
        free(hsum);
        return;
    }
    for (long i = 0; i < n; ++i) {
        long flat = tokens ? (long)tokens[i] : i;
        int s = (int)(flat / T);
        const int32_t *ids = topk_ids + (size_t)flat * K;
        size_t o = (size_t)i * H;

        /* which rank's message sits in which slot (first occurrence wins) */
        for (int k = 0; k < P; ++k) {
            slot_dest[k] = -1;
            if (k >= K || ids[k] < 0 || ids[k] >= E)
                continue;
            int d = ids[k] / Epr;
            int earlier = 0;
            for (int k2 = 0; k2 < k; ++k2)
                if (ids[k2] >= 0 && ids[k2] < E && ids[k2] / Epr == d)
                    earlier = 1;
            if (!earlier)
                slot_dest[k] = d;
        }

        for (int h = 0; h < H; ++h) {
            for (int k = 0; k < P; ++k) {
                a[k] = 0.0f;
                if (slot_dest[k] >= 0) {
                    int d = slot_dest[k];
                    int32_t j = send_slot[(size_t)flat * R + d];
                    size_t row = ((size_t)d * R + s) * m + (size_t)j;
                    a[k] = oracle_f32_from_bf16(expert_out[row * H + h]);
                }
            }
            for (int stride = 1; stride < P; stride *= 2)
                for (int k = 0; k + stride < P; k += 2 * stride)
                    a[k] = oracle_f32_from_bf16(oracle_bf16_from_f32(a[k] + a[k + stride]));
            acc[h] = a[0];
        }
        finish_row(H, acc, residual ? residual + (size_t)flat * H : 0, gamma, eps, hsum,
                   out + o, residual_out ? residual_out + o : 0, y_ref ? y_ref + o : 0);
    }
    free(slot_dest);
    free(a);
    free(acc);
    free(hsum);
}

/* ------------------------------------------------------------------------ */
/* Expert-major layout: every received row carries one expert                */
/* ------------------------------------------------------------------------ */

/*
 * [IX] "Best remaining lead" (the association-order analysis): backends
 * whose received rows each carry a single expert -- the low-latency padded
 * layouts -- never meet the per-rank aggregation question; [IX] review of
 * the harness: those backends declare "weighted-kernel-sum", the gates
 * being applied by the combine kernel, and the oracle's message sums the
 * top-k axis in problem order.  Readings (the pages name the layout, not its
 * arithmetic):
 *   - expert e has a plane of cap = R * m rows; one row per distinct
 *     (token, expert) with 0 <= e < E, in ascending (source rank, token);
 *   - send_row[s][t][k] = e_k * cap + slot for the first k with that expert,
 *     -1 for a later duplicate or an id outside [0, E);
 *   - wsum[s][t][k] = sum over the token's k' with the same expert, in
 *     ascending k', of w[k'] from +0.0f (first occurrence; 0.0f elsewhere);
 *   - recv_counts[e] = rows of expert e; src_row[e][j] = s * T + t of row j
 *     (-1 past the count); recv_w[e][j] = the row's wsum;
 *   - local_expert_counts[e] counts valid (token, k) entries, duplicates
 *     included, as in the rank layout.
 * Returns the number of ids outside [-1, E).
 */
long oracle_route_experts(int R, int T, int K, int E, int m,
                          const int32_t *topk_ids, const float *topk_w,
                          int32_t *send_row, float *wsum, int32_t *recv_counts,
                          int32_t *src_row, float *recv_w, int32_t *local_expert_counts)
{
    const long cap = (long)R * m;
    long invalid = 0;
    for (int e = 0; e < E; ++e) {
        recv_counts[e] = 0;
        local_expert_counts[e] = 0;
    }
    for (long i = 0; i < (long)E * cap; ++i) {
        src_row[i] = -1;
        recv_w[i] = 0.0f;
    }
    /* sources in ascending order, tokens in ascending order: each distinct
       expert of a token takes the next row of that expert's plane */
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < T; ++t) {
            long flat = (long)s * T + t;
            const int32_t *ids = topk_ids + (size_t)flat * K;
            const float *w = topk_w + (size_t)flat * K;
            for (int k = 0; k < K; ++k) {
                int32_t e = ids[k];
                send_row[(size_t)flat * K + k] = -1;
                wsum[(size_t)flat * K + k] = 0.0f;
                if (e == -1)
                    continue;
                if (e < -1 || e >= E) {
                    invalid += 1;
                    continue;
                }
                local_expert_counts[e] += 1;
                int first = 1;
                for (int k2 = 0; k2 < k; ++k2)
                    if (ids[k2] == e)
                        first = 0;
                if (!first)
                    continue;
                float sum = 0.0f;
                for (int k2 = k; k2 < K; ++k2)
                    if (ids[k2] == e)
                        sum = sum + w[k2];
                long j = recv_counts[e];
                recv_counts[e] += 1;
                send_row[(size_t)flat * K + k] = (int32_t)(e * cap + j);
                wsum[(size_t)flat * K + k] = sum;
                src_row[e * cap + j] = (int32_t)flat;
                recv_w[e * cap + j] = sum;
            }
        }
    }
    return invalid;
}

/*
 * recv_x [E][cap][H] bf16: row j of expert e = x[src_row[e][j]]; only rows
 * j < recv_counts[e] are written.
 */
void oracle_dispatch_experts(int R, int E, int H, int m, const uint16_t *x,
                             const int32_t *recv_counts, const int32_t *src_row,
                             uint16_t *recv_x)
{
    const long cap = (long)R * m;
    for (int e = 0; e < E; ++e) {
        for (int j = 0; j < recv_counts[e]; ++j) {
            long flat = src_row[e * cap + j];
            for (int h = 0; h < H; ++h)
                recv_x[((size_t)e * cap + j) * H + h] = x[(size_t)flat * H + h];
        }
    }
}

/*
 * For each requested token (flat s*T + t; tokens == NULL means all):
 *   acc[h] = sum over k ascending with send_row[s][t][k] >= 0 of
 *            v = f32(expert_out[send_row][h])                   (weighted=0)
 *            wsum[s][t][k] * v                                   (weighted=1)
 *            from +0.0f, one fp32 multiply and one fp32 add each
 * ("weighted-kernel-sum" in problem order), then the epilogue of
 * finish_row.  expert_out is [E][cap][H] bf16.
 */
void oracle_combine_experts(int R, int T, int K, int H, int weighted,
                            const int32_t *send_row, const float *wsum,
                            const uint16_t *expert_out, const uint16_t *residual,
                            const uint16_t *gamma, float eps,
                            const int64_t *tokens, long ntokens,
                            float *acc_out, uint16_t *out, uint16_t *residual_out,
                            double *y_ref)
{
    long n = tokens ? ntokens : (long)R * T;
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    float *hsum = (float *)malloc((size_t)H * sizeof(float));
    if (!acc || !hsum) {
        free(acc);
        free(hsum);
        return;
    }
    for (long i = 0; i < n; ++i) {
        long flat = tokens ? (long)tokens[i] : i;
        size_t o = (size_t)i * H;
        for (int h = 0; h < H; ++h) {
            float a = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t row = send_row[(size_t)flat * K + k];
                if (row < 0)
                    continue;
                float v = oracle_f32_from_bf16(expert_out[(size_t)row * H + h]);
                if (weighted) {
                    float p = wsum[(size_t)flat * K + k] * v;
                    a = a + p;
                } else {
                    a = a + v;
                }
            }
            acc[h] = a;
            if (acc_out)
                acc_out[o + h] = a;
        }
        finish_row(H, acc, residual ? residual + (size_t)flat * H : 0, gamma, eps, hsum,
                   out + o, residual_out ? residual_out + o : 0, y_ref ? y_ref + o : 0);
    }
    free(acc);
    free(hsum);
}

/* ------------------------------------------------------------------------ */
/* Expert-side consumer of the expert planes: a grouped matrix product       */
/* ------------------------------------------------------------------------ */

/*
 * [IX] "Why" / the harness review: between dispatch and combine each
 * expert applies its own weights to the rows it received (vLLM applies the
 * gates in the MoE layer, around this product).  Reading: one linear map per
 * expert, W_e of N x H (row n holds the weights of output n, as a linear
 * layer stores them), applied to every received row of that expert:
 *   y[e][j][n] = sum over h of f32(x[e][j][h]) * f32(w[e][n][h])
 * for j < recv_counts[e], taken here in double (the exact value of the sum of
 * the bf16 products, up to double rounding); rows j >= recv_counts[e] of y
 * are not written.  x is [E][cap][H] bf16, w [E][N][H] bf16, y [E][cap][N].
 */
void oracle_expert_gemm(int E, long cap, int H, int N, const int32_t *recv_counts,
                        const uint16_t *x, const uint16_t *w, double *y)
{
    for (int e = 0; e < E; ++e) {
        for (long j = 0; j < recv_counts[e]; ++j) {
            const uint16_t *xr = x + ((size_t)e * cap + j) * H;
            for (int n = 0; n < N; ++n) {
                const uint16_t *wr = w + ((size_t)e * N + n) * H;
                double acc = 0.0;
                for (int h = 0; h < H; ++h)
                    acc += (double)oracle_f32_from_bf16(xr[h]) * (double)oracle_f32_from_bf16(wr[h]);
                y[((size_t)e * cap + j) * N + n] = acc;
            }
        }
    }
}

/*
 * The same expert-side product on the rank planes (the receive layout the
 * rank dispatch produces).  A received row (d, s, j) carries one token and
 * the token's experts that live on rank d (recv_ids, -1 elsewhere).  [IX]
 * "Why": each expert applies its weights to the rows it received; vLLM
 * applies the gates in the MoE layer, so rank d's message for the token is
 * its experts' outputs summed with their gates.  Readings (the pages give no
 * arithmetic): the output of expert e_k on the row is a bf16 value,
 *   y_k[n] = bf16_rn(f32_rn(sum_h x[h] * w[e_k][n][h]))   (the sum exact here,
 *            in double, then rounded to binary32 and to bf16),
 * and the row's message is
 *   msg[n] = bf16_rn(sum over k ascending with recv_ids[k] >= 0 of
 *                    g_k * y_k[n]),  g_k = recv_w[k] (apply_gates) or 1,
 * in binary32 from +0.0, one multiply and one add per term (no FMA).
 * Only rows j < recv_counts[d][s] are computed, or only the flat rows
 * (d * R + s) * m + j listed in `rows` (n_rows of them) when rows != NULL;
 * msg is [R][R][m][N] (other rows untouched).  ymag / smag (optional, same
 * shape, double) receive the magnitudes sum_k |g_k| |y_k exact| and
 * sum_k |g_k| sum_h |x[h] w[e_k][n][h]| that bound rounding differences.
 */
void oracle_expert_gemm_rank(int R, int m, int K, int H, int N, const int32_t *recv_counts,
                             const uint16_t *recv_x, const int32_t *recv_ids,
                             const float *recv_w, const uint16_t *w, int apply_gates,
                             const int64_t *rows, long n_rows, uint16_t *msg, double *ymag,
                             double *smag)
{
    long total = rows != NULL ? n_rows : (long)R * R * m;
    for (long i = 0; i < total; ++i) {
        long flat = rows != NULL ? (long)rows[i] : i;
        long plane = flat / m;
        long j = flat - plane * m;
        int d = (int)(plane / R), s = (int)(plane % R);
        if (d >= R || j >= recv_counts[d * R + s])
            continue;
        const uint16_t *xr = recv_x + (size_t)flat * H;
        const int32_t *ids = recv_ids + (size_t)flat * K;
        const float *g = recv_w + (size_t)flat * K;
        for (int n = 0; n < N; ++n) {
            float a = 0.0f;
            double ym = 0.0, sm = 0.0;
            for (int k = 0; k < K; ++k) {
                int e = ids[k];
                if (e < 0)
                    continue;
                const uint16_t *wr = w + ((size_t)e * N + n) * H;
                double y = 0.0, mag = 0.0;
                for (int h = 0; h < H; ++h) {
                    double prod = (double)oracle_f32_from_bf16(xr[h]) *
                                  (double)oracle_f32_from_bf16(wr[h]);
                    y += prod;
                    mag += fabs(prod);
                }
                float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));
                float gk = apply_gates ? g[k] : 1.0f;
                float p = gk * yk;
                a = a + p;
                ym += fabs((double)gk) * fabs(y);
                sm += fabs((double)gk) * mag;
            }
            msg[(size_t)flat * N + n] = oracle_bf16_from_f32(a);
            if (ymag != NULL)
                ymag[(size_t)flat * N + n] = ym;
            if (smag != NULL)
                smag[(size_t)flat * N + n] = sm;
        }
    }
}

/* forward declaration: the e4m3 decoding defined with the FP8 helpers below */
float oracle_f32_from_fp8e4m3(uint8_t q);

/*
 * The same product on FP8 operands: the rows as the FP8 receive format holds
 * them (e4m3 codes qx with one scale sx per row) and weights as e4m3 codes qw
 * with one scale sw per output channel.  Reading (the pages name FP8
 * payloads with a scale payload, not this arithmetic): dequantised operands,
 *   y[e][j][n] = sx[e][j] * sw[e][n] * sum_h f(qx[e][j][h]) * f(qw[e][n][h]),
 * f the e4m3 value; the sum and the scaling in double here.  Rows past a
 * count are not written.  qx [E][cap][H], sx [E][cap], qw [E][N][H], sw [E][N].
 */
void oracle_expert_gemm_fp8(int E, long cap, int H, int N, const int32_t *recv_counts,
                            const uint8_t *qx, const float *sx, const uint8_t *qw,
                            const float *sw, double *y)
{
    for (int e = 0; e < E; ++e) {
        for (long j = 0; j < recv_counts[e]; ++j) {
            const uint8_t *xr = qx + ((size_t)e * cap + j) * H;
            for (int n = 0; n < N; ++n) {
                const uint8_t *wr = qw + ((size_t)e * N + n) * H;
                double acc = 0.0;
                for (int h = 0; h < H; ++h)
                    acc += (double)oracle_f32_from_fp8e4m3(xr[h]) * (double)oracle_f32_from_fp8e4m3(wr[h]);
                y[((size_t)e * cap + j) * N + n] =
                    (double)sx[(size_t)e * cap + j] * (double)sw[(size_t)e * N + n] * acc;
            }
        }
    }
}

/*
 * The product on the rank planes with FP8 operands: the received rows as the
 * FP8 receive format holds them (e4m3 codes qx, one scale sx per received
 * row), the weights as e4m3 codes qw with one scale sw per output channel.
 * Readings: as oracle_expert_gemm_rank, with each expert output formed from
 * the dequantised operands as in oracle_expert_gemm_fp8,
 *   y_k[n] = bf16_rn(f32_rn(sx * sw[e_k][n] * sum_h f(qx[h]) * f(qw[e_k][n][h])))
 * (the product and the scaling exact here, in double), then
 *   msg[n] = bf16_rn(sum over k ascending with recv_ids[k] >= 0 of g_k * y_k[n])
 * in binary32 from +0.0, one multiply and one add per term.  recv_x8
 * [R][R][m][H] codes, recv_scale [R][R][m], qw [E][N][H], sw [E][N]; rows,
 * msg, ymag and smag as in oracle_expert_gemm_rank (the magnitudes include
 * |sx sw|).
 */
void oracle_expert_gemm_rank_fp8(int R, int m, int K, int H, int N,
                                 const int32_t *recv_counts, const uint8_t *recv_x8,
                                 const float *recv_scale, const int32_t *recv_ids,
                                 const float *recv_w, const uint8_t *qw, const float *sw,
                                 int apply_gates, const int64_t *rows, long n_rows,
                                 uint16_t *msg, double *ymag, double *smag)
{
    long total = rows != NULL ? n_rows : (long)R * R * m;
    for (long i = 0; i < total; ++i) {
        long flat = rows != NULL ? (long)rows[i] : i;
        long plane = flat / m;
        long j = flat - plane * m;
        int d = (int)(plane / R), s = (int)(plane % R);
        if (d >= R || j >= recv_counts[d * R + s])
            continue;
        const uint8_t *xr = recv_x8 + (size_t)flat * H;
        const double sx = (double)recv_scale[flat];
        const int32_t *ids = recv_ids + (size_t)flat * K;
        const float *g = recv_w + (size_t)flat * K;
        for (int n = 0; n < N; ++n) {
            float a = 0.0f;
            double ym = 0.0, sm = 0.0;
            for (int k = 0; k < K; ++k) {
                int e = ids[k];
                if (e < 0)
                    continue;
                const uint8_t *wr = qw + ((size_t)e * N + n) * H;
                const double scale = sx * (double)sw[(size_t)e * N + n];
                double acc = 0.0, mag = 0.0;
                for (int h = 0; h < H; ++h) {
                    double prod = (double)oracle_f32_from_fp8e4m3(xr[h]) *
                                  (double)oracle_f32_from_fp8e4m3(wr[h]);
                    acc += prod;
                    mag += fabs(prod);
                }
                double y = scale * acc;
                float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));
                float gk = apply_gates ? g[k] : 1.0f;
                float p = gk * yk;
                a = a + p;
                ym += fabs((double)gk) * fabs(y);
                sm += fabs((double)gk) * fabs(scale) * mag;
            }
            msg[(size_t)flat * N + n] = oracle_bf16_from_f32(a);
            if (ymag != NULL)
                ymag[(size_t)flat * N + n] = ym;
            if (smag != NULL)
                smag[(size_t)flat * N + n] = sm;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 (OCP e4m3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no  */
/* infinity, NaN = S.1111.111, largest finite 448) and per-token scaling     */
/* ------------------------------------------------------------------------ */

/* Widening is exact: exponent field 0 holds subnormals m * 2^-9. */
float oracle_f32_from_fp8e4m3(uint8_t q)
{
    int sign = (q >> 7) & 1;
    int e = (q >> 3) & 0xf;
    int m = q & 7;
    float v;
    if (e == 0xf && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexpf((float)m, -9);
    else
        v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return sign ? -v : v;
}

/* Narrowing with round-to-nearest, ties-to-even, saturating to +-448
 * (magnitudes above the largest finite value become 448); NaN stays NaN.
 * Works on the binary32 bit pattern: the kept bits are the leading
 * significand bits that fit the target exponent (3 below the leading 1 for
 * normals, fewer for subnormals); the dropped bits are compared with one
 * half of the kept unit. */
uint8_t oracle_fp8e4m3_from_f32(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    uint32_t exp32 = (bits >> 23) & 0xffu;
    uint32_t man32 = bits & 0x7fffffu;
    if (exp32 == 0xffu && man32 != 0u)
        return (uint8_t)(sign | 0x7f);
    if (exp32 == 0xffu || fabsf(f) > 448.0f)
        return (uint8_t)(sign | 0x7e);
    if (exp32 == 0u)            /* binary32 zero or subnormal: below 2^-126 */
        return sign;
    /* value = 1.man32 * 2^(exp32 - 127); count in units of the target ulp */
    int e = (int)exp32 - 127;
    int ulp_exp = e >= -6 ? e - 3 : -9;          /* exponent of the kept unit */
    uint64_t sig = (uint64_t)(0x800000u | man32); /* times 2^(e - 23) */
    int shift = ulp_exp - (e - 23);              /* bits dropped */
    if (shift >= 64)           /* far below half of the smallest subnormal */
        return sign;
    uint64_t kept = sig >> shift;
    uint64_t dropped = sig & (((uint64_t)1 << shift) - 1);
    uint64_t half = (uint64_t)1 << (shift - 1);
    if (dropped > half || (dropped == half && (kept & 1u)))
        kept += 1;
    /* kept counts units of 2^ulp_exp: rebuild the code */
    if (e < -6) {
        /* subnormal units of 2^-9; 8 units is the smallest normal, code 0x08 */
        return (uint8_t)(sign | (uint8_t)kept);
    }
    /* normal: kept in [8, 16]; 16 means the next binade */
    int ee = e;
    if (kept == 16) {
        kept = 8;
        ee += 1;
    }
    if (ee > 8 || (ee == 8 && kept > 14))
        return (uint8_t)(sign | 0x7e);               /* saturate */
    return (uint8_t)(sign | (uint8_t)(((ee + 7) << 3) | (uint8_t)(kept - 8)));
}

/* Per-token FP8 quantisation of bf16 rows [n][H]: amax = max_h |x_h|
 * (binary32, exact), scale = amax / 448 (one binary32 division; 1 when the
 * row is all zero), q_h = fp8(x_h / scale) (one binary32 division, then the
 * narrowing above).  Dequantised value: f32(q_h) * scale. */
void oracle_quantize_rows_fp8(long n, int H, const uint16_t *x, uint8_t *q, float *scale)
{
    for (long i = 0; i < n; ++i) {
        const uint16_t *row = x + (size_t)i * H;
        float amax = 0.0f;
        for (int h = 0; h < H; ++h) {
            float a = fabsf(oracle_f32_from_bf16(row[h]));
            if (a > amax)
                amax = a;
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[i] = sc;
        for (int h = 0; h < H; ++h)
            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(oracle_f32_from_bf16(row[h]) / sc);
    }
}

/* The same for binary32 rows (the combine's output before narrowing). */
void oracle_quantize_f32_rows_fp8(long n, int H, const float *x, uint8_t *q, float *scale)
{
    for (long i = 0; i < n; ++i) {
        const float *row = x + (size_t)i * H;
        float amax = 0.0f;
        for (int h = 0; h < H; ++h)
            if (fabsf(row[h]) > amax)
                amax = fabsf(row[h]);
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[i] = sc;
        for (int h = 0; h < H; ++h)
            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(row[h] / sc);
    }
}

