// dispatch.cu -- scatter of token rows into the padded receive planes.
//
// Operation (InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided
// NVLink EP for the GB SKUs": "Why" -- the initiator writes the token row
// straight into the target's workspace; "The adapter" -- receive is padded
// [ep_size, runtime_max_tokens_per_rank, hidden] and only valid slots are
// meaningful):
//   recv_x[d][s][slot(s,t,d)][:] = x[s][t][:]   for every d in dmask(s,t).
// Padding slots are never written.
//
// GB300 design: the row is read from HBM once and written once per
// destination.  Each CTA is one warp whose lane 0 drives a ring of shared
// memory stages with 1-D bulk asynchronous copies: a bulk load brings the
// row chunk and the token's send-slot row into a stage (completion counted
// on the stage's mbarrier), then one bulk store per destination writes the
// chunk out of shared memory.  Launched straight after the first routing
// pass (rank layout), the send-slot row holds the token's slots inside its
// routing tile and a third bulk load brings the tile's exclusive prefix
// row; their sum is the slot, so the copy does not wait for the second
// pass, which runs beside it.  Stages are refilled one iteration after
// their stores were issued, so S-1 loads stay in flight per CTA while the
// stores drain.  The copy engine moves every byte; the thread only issues.
// Waits are bounded: if one runs out the kernel raises the timeout flag,
// drains its copies and returns.
#include "kernels.h"
#include "ptx.cuh"
#include "smem_limit.h"

#include "moe_a2a.h"

namespace moe {
namespace {

constexpr uint32_t kWaitLimit = 1u << 24;  // try_wait probes before giving up
constexpr int kMaxChunk = 16384;

__global__ void __launch_bounds__(32) dispatch_rows_kernel(const DispatchParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)p.stages * p.stage_bytes);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) ptx::mbar_init(&bars[i], 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x != 0) {
        ptx::grid_dependency_wait();
        return;
    }

    const long long first = blockIdx.x, step = gridDim.x;
    const long long n = first < p.units ? (p.units - 1 - first) / step + 1 : 0;
    const uint32_t meta_bytes = (uint32_t)p.dest.P * 4u;
    const bool split = p.tile_prefix != nullptr;  // local slots + tile prefixes

    auto unit_bytes = [&](int chunk) -> uint32_t {
        const int left = p.row_bytes - chunk * p.chunk_bytes;
        return (uint32_t)(left < p.chunk_bytes ? left : p.chunk_bytes);
    };
    // Unit i of this CTA: a chunk of the row of token (s, t), stored at row
    // s * stride + t of the token arrays.
    auto unit_of = [&](long long i, int &s, long long &row, int &chunk, int &t) {
        const long long u = first + i * step;
        // rows up to 16 KB (H <= 8192) are one chunk: no division on the
        // issuing lane's path
        const long long k = p.chunks == 1 ? u : u / p.chunks;
        chunk = (int)(u - k * p.chunks);
        token_of(p.map, p.R, k, s, t);
        row = (long long)s * p.map.stride + t;
    };
    // A unit's stage receives its row chunk (an input of the call) and its
    // send row (written by the routing pass); both complete on one barrier.
    auto issue_row = [&](long long i, int stage) {  // stage = i mod stages
        int s, chunk, t;
        long long token;
        unit_of(i, s, token, chunk, t);
        uint8_t *buf = smem + (size_t)stage * p.stage_bytes;
        const uint32_t bytes = unit_bytes(chunk);
        ptx::fence_proxy_async_smem();  // earlier ordinary reads of this stage
        ptx::mbar_arrive_expect_tx(&bars[stage], bytes + (split ? 2 : 1) * meta_bytes);
        ptx::bulk_g2s(buf, p.x + token * p.row_bytes + (long long)chunk * p.chunk_bytes, bytes,
                      &bars[stage]);
    };
    auto issue_meta = [&](long long i, int stage) {
        int s, chunk, t;
        long long token;
        unit_of(i, s, token, chunk, t);
        uint8_t *buf = smem + (size_t)stage * p.stage_bytes;
        ptx::bulk_g2s(buf + p.chunk_bytes, p.send_slot + token * p.dest.P, meta_bytes,
                      &bars[stage]);
        if (split)  // the exclusive prefix of the token's tile, per destination
            ptx::bulk_g2s(buf + p.chunk_bytes + meta_bytes,
                          p.tile_prefix + ((long long)s * p.ntiles + t / p.tile) * p.dest.P,
                          meta_bytes, &bars[stage]);
    };
    auto issue = [&](long long i, int stage) {
        issue_row(i, stage);
        issue_meta(i, stage);
    };

    // The first stages' rows are in flight while the routing pass finishes.
    const long long prologue = n < p.stages ? n : p.stages;
    for (long long i = 0; i < prologue; ++i) issue_row(i, (int)i);
    ptx::grid_dependency_wait();  // send-slot table of the routing pass
    for (long long i = 0; i < prologue; ++i) issue_meta(i, (int)i);
    long long issued = prologue;

    // stage = i mod stages and the barrier parity, stepped along with i
    int stage = 0, prev_stage = p.stages - 1;
    uint32_t parity = 0;
    for (long long i = 0; i < n; ++i) {
        if (!ptx::mbar_wait_bounded(&bars[stage], parity, kWaitLimit)) {
            atomicOr(p.flags, MOE_DEVICE_FLAG_WAIT_TIMEOUT);
            ptx::bulk_wait_all();
            for (long long j = i + 1; j < issued; ++j)
                ptx::mbar_wait_bounded(&bars[j % p.stages], (uint32_t)((j / p.stages) & 1),
                                       kWaitLimit);
            return;
        }
        int s, chunk, t;
        long long token;
        unit_of(i, s, token, chunk, t);
        uint8_t *buf = smem + (size_t)stage * p.stage_bytes;
        const int32_t *slots = reinterpret_cast<const int32_t *>(buf + p.chunk_bytes);
        const int32_t *prefix = slots + p.dest.P;
        const uint32_t bytes = unit_bytes(chunk);
        const long long col = (long long)chunk * p.chunk_bytes;
        for (int d = 0; d < p.dest.P; ++d) {
            const int32_t slot = slots[d] < 0 ? -1 : slots[d] + (split ? prefix[d] : 0);
            if (slot < 0) continue;
            const long long row = dest_row(p.dest, p.R, p.m, d, s, slot);
            if (row < 0) {  // guard: never expected from the routing pass
                atomicOr(p.flags, MOE_DEVICE_FLAG_BAD_SLOT);
                continue;
            }
            ptx::bulk_s2g(p.recv_x + row * p.row_bytes + col, buf, bytes);
        }
        ptx::bulk_commit();
        // Refill the stage of iteration i-1 once its stores left shared memory
        // (issued = i - 1 + stages: that stage).
        if (i >= 1 && issued < n) {
            ptx::bulk_wait_read<1>();
            issue(issued, prev_stage);
            ++issued;
        }
        prev_stage = stage;
        if (++stage == p.stages) {
            stage = 0;
            parity ^= 1u;
        }
    }
    ptx::bulk_wait_all();
}

}  // namespace

cudaError_t dispatch_prepare(int row_bytes, int P, int num_sms, const Tuning &tn,
                             DispatchParams *p, LaunchShape *shape) {
    const int chunks = (row_bytes + kMaxChunk - 1) / kMaxChunk;
    int chunk = (row_bytes + chunks - 1) / chunks;
    chunk = (chunk + 15) / 16 * 16;
    const int stage_bytes = (chunk + 2 * P * 4 + 127) / 128 * 128;  // row, slots, prefixes
    int stages = 65536 / stage_bytes;
    stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    if (tn.dispatch_stages > 0) stages = tn.dispatch_stages;
    const size_t smem = (size_t)stages * stage_bytes + (size_t)stages * sizeof(uint64_t);

    cudaError_t err = raise_smem_limit(dispatch_rows_kernel, smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_rows_kernel, 32, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (tn.dispatch_ctas_per_sm > 0) per_sm = tn.dispatch_ctas_per_sm;

    p->row_bytes = row_bytes;
    p->chunk_bytes = chunk;
    p->chunks = chunks;
    p->stages = stages;
    p->stage_bytes = stage_bytes;
    shape->grid = num_sms * per_sm;
    shape->block = 32;
    shape->smem = smem;
    return cudaSuccess;
}

cudaError_t launch_dispatch_rows(const DispatchParams &p, const LaunchShape &shape,
                                 cudaStream_t st, bool pdl) {
    long long grid = shape.grid;
    if (grid > p.units) grid = p.units;
    if (grid < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = shape.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, dispatch_rows_kernel, p);
}

}  // namespace moe
