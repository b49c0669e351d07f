// moe_noalloc.cu -- the routing pass with its scratch in a fixed device
// array, for callers that cannot allocate device memory.
//
// Who needs this: code that runs inside a host framework which owns every
// byte of device memory and hands out no allocator (a plugin or custom op
// in an inference engine), and serving loops that forbid device allocation
// after start-up because cudaMalloc can synchronise the whole device and
// fragments a fixed memory budget.  Such callers can still pass their own
// input and output buffers; what they cannot do is provide the routing
// pass's temporary working memory.  Here that memory is a file-scope
// __device__ array that the CUDA runtime creates when the library is loaded
// on a device and keeps until the process exits.
//
// The entry point runs the same two routing kernels as moe_dispatch
// (route_count, route_scan); only the source of their scratch differs.
#include "moe_a2a.h"

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace {

// A CUDA call of this library failed.  The status says so; the runtime's
// last error, which a refused launch also leaves behind, is cleared so that
// the caller's next, unrelated CUDA call does not report it again.
int cuda_failed() {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
}

constexpr size_t kScratchBytes = MOE_STATIC_SCRATCH_BYTES;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

// The scratch: per-tile destination counts and prefixes (tiles of 256
// tokens), per-source tickets, per-source expert histograms, and one
// word that absorbs device flags when the caller passes no flag output.
// Shared by every call on a device.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

// The array's device address belongs to the context that loaded the module:
// a device reset (cudaDeviceReset, or a framework that tears down and
// recreates the primary context) reloads the module, possibly elsewhere.  So
// the address is kept together with the driver's unique id of the context it
// was looked up in, and looked up again whenever the current context differs.
struct ScratchSlot {
    unsigned long long ctx_id;  // 0: never looked up
    void *addr;
};

std::mutex g_mutex;
ScratchSlot g_slot[kMaxDevices];

// Driver entry points reached through the runtime (no link against the
// driver library): the current context and its process-unique id.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

bool resolve_driver_calls() {  // under g_mutex
    if (g_ctx_get_current != nullptr && g_ctx_get_id != nullptr) return true;
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) !=
            cudaSuccess ||
        qa != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess ||
        qb != cudaDriverEntryPointSuccess || a == nullptr || b == nullptr)
        return false;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
    return true;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of g_route_scratch in the current context (host code cannot
// use the symbol itself as a device pointer).  Looked up with
// cudaGetSymbolAddress the first time a context is seen; that lookup is not
// made while `st` is capturing (it can load the module), which returns
// MOE_ERR_SETUP_IN_CAPTURE instead.
int scratch_address(cudaStream_t st, void **out) {
    // A runtime call that needs the context first, so that the device's
    // primary context exists and is current before it is queried.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return cuda_failed();
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cuda_failed();
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!resolve_driver_calls()) return cuda_failed();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        g_ctx_get_id(ctx, &id) != CUDA_SUCCESS || id == 0)
        return cuda_failed();
    ScratchSlot &slot = g_slot[dev];
    if (slot.ctx_id != id) {
        if (cap != cudaStreamCaptureStatusNone) return MOE_ERR_SETUP_IN_CAPTURE;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
            return cuda_failed();
        slot.addr = p;
        slot.ctx_id = id;
    }
    *out = slot.addr;
    return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" size_t moe_route_static_scratch_bytes(int32_t ep_size, int32_t num_experts,
                                                 int32_t tokens_per_rank) {
    if (ep_size < 1 || num_experts < 1 || tokens_per_rank < 0) return 0;
    const size_t R = ep_size, E = num_experts, T = tokens_per_rank;
    const size_t RP = (R + 3) / 4 * 4;
    const size_t tiles = (T + moe::kRouteTile - 1) / moe::kRouteTile;
    return 2 * align_up(R * tiles * RP * 4, kAlign) + align_up(R * 4 + R * E * 4, kAlign) +
           kAlign;
}

extern "C" int moe_route_static_scratch(int32_t ep_size, int32_t num_experts, int32_t top_k,
                                        int32_t tokens_per_rank,
                                        int32_t runtime_max_tokens_per_rank,
                                        const int32_t *d_topk_ids, const float *d_topk_w,
                                        int32_t *d_send_slot, float *d_dest_weight,
                                        int32_t *d_src_token, int32_t *d_recv_counts,
                                        int32_t *d_local_expert_counts,
                                        int32_t *d_recv_topk_ids, float *d_recv_topk_w,
                                        uint32_t *d_flags, void *stream) {
    const int R = ep_size, E = num_experts, K = top_k, T = tokens_per_rank;
    const int m = runtime_max_tokens_per_rank;
    if (R < 1 || R > MOE_MAX_EP_SIZE || E < R || E > MOE_MAX_EXPERTS || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (K < 1 || K > MOE_MAX_TOP_K || T < 0 || m < 1) return MOE_ERR_INVALID_ARG;
    if (T > m) return MOE_ERR_CAPACITY;
    if (moe_route_static_scratch_bytes(R, E, T) > kScratchBytes) return MOE_ERR_CAPACITY;
    if (d_recv_counts == nullptr || d_local_expert_counts == nullptr) return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (d_topk_ids == nullptr || d_topk_w == nullptr || d_send_slot == nullptr ||
            d_dest_weight == nullptr || d_src_token == nullptr || d_recv_topk_ids == nullptr ||
            d_recv_topk_w == nullptr)
            return MOE_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(d_topk_ids) & 3u) ||
            (reinterpret_cast<uintptr_t>(d_topk_w) & 3u) || !aligned16(d_send_slot) ||
            !aligned16(d_dest_weight) || !aligned16(d_src_token) ||
            !aligned16(d_recv_topk_ids) || !aligned16(d_recv_topk_w))
            return MOE_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (T == 0) {
        if (cudaMemsetAsync(d_recv_counts, 0, sizeof(int32_t) * R * R, st) != cudaSuccess ||
            cudaMemsetAsync(d_local_expert_counts, 0, sizeof(int32_t) * E, st) != cudaSuccess)
            return cuda_failed();
        return MOE_OK;
    }

    void *base = nullptr;
    const int rc = scratch_address(st, &base);
    if (rc != MOE_OK) return rc;

    // Carve the scratch: per-tile counts and prefixes (written before they
    // are read in this call), then the per-source tickets and the expert
    // histogram accumulator, which must start at zero and are cleared here.
    const int RP = (R + 3) / 4 * 4;
    const int ntiles = (T + moe::kRouteTile - 1) / moe::kRouteTile;
    unsigned char *p = static_cast<unsigned char *>(base);
    int32_t *tile_counts = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)R * ntiles * RP * 4, kAlign);
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)R * ntiles * RP * 4, kAlign);
    int32_t *tile_ticket = reinterpret_cast<int32_t *>(p);
    int32_t *hist_accum = tile_ticket + R;
    if (cudaMemsetAsync(tile_ticket, 0, sizeof(int32_t) * ((size_t)R + (size_t)R * E), st) !=
        cudaSuccess)
        return cuda_failed();
    p += align_up((size_t)R * 4 + (size_t)R * E * 4, kAlign);
    uint32_t *sink_flags = reinterpret_cast<uint32_t *>(p);

    moe::TokenMap map;
    map.stride = T;
    map.uniform = 1;
    for (int r = 0; r < moe::kMaxRanks; ++r) {
        map.count[r] = r < R ? T : 0;
        map.first[r] = (r < R ? r : R) * T;
    }
    map.first[moe::kMaxRanks] = R * T;
    const uint32_t all = R >= 32 ? 0xffffffffu : ((1u << R) - 1u);

    moe::RouteCountParams c;
    c.topk_ids = d_topk_ids;
    c.tile_counts = tile_counts;
    c.tile_prefix = tile_prefix;
    c.local_slot = nullptr;
    c.tile_ticket = tile_ticket;
    c.hist_accum = hist_accum;
    c.recv_counts = d_recv_counts;
    c.flags = d_flags != nullptr ? d_flags : sink_flags;
    c.map = map;
    c.active = all;
    c.R = R, c.K = K, c.E = E, c.Epr = E / R, c.RP = RP, c.ntiles = ntiles;
    c.tile = moe::kRouteTile;
    if (moe::launch_route_count(c, st) != cudaSuccess) return cuda_failed();

    moe::RouteScanParams s;
    s.topk_ids = d_topk_ids;
    s.topk_w = d_topk_w;
    s.tile_prefix = tile_prefix;
    s.hist_accum = hist_accum;
    s.send_slot = d_send_slot;
    s.dest_weight = d_dest_weight;
    s.src_token = d_src_token;
    s.recv_ids = d_recv_topk_ids;
    s.recv_w = d_recv_topk_w;
    s.topk_dest = nullptr;
    s.local_counts = d_local_expert_counts;
    s.map = map;
    s.active = all;
    s.R = R, s.K = K, s.E = E, s.Epr = E / R, s.RP = RP, s.m = m, s.ntiles = ntiles;
    s.tile = moe::kRouteTile;
    s.dg = 4;
    if (moe::launch_route_scan(s, st, true) != cudaSuccess) return cuda_failed();
    return MOE_OK;
}
