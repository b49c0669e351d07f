"""The allocation-free routing entry point, checked against moe_dispatch.

moe_route_static_scratch serves callers that cannot allocate device memory
(a plugin inside a framework that owns the memory pool, a serving loop that
forbids cudaMalloc after start-up): they pass inputs and outputs, and the
routing pass's temporary memory is the library's fixed device array.  Its
outputs must equal the ones moe_dispatch produces for the same routing,
bit for bit (integer and copied data), on consecutive calls that reuse the
shared array.  This file is collected last on purpose.
"""
import numpy as np
import pytest

from combine_topk_ids_rank_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module")
def mod():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()
    from combine_topk_ids_rank_gb300 import moe_a2a
    return moe_a2a


def static_route(mod, R, E, K, T, m, ids, w):
    RP = (R + 3) // 4 * 4
    dev = ids.device
    out = dict(send_slot=torch.full((R, T, RP), -7, dtype=torch.int32, device=dev),
               dest_weight=torch.full((R, T, RP), -7.0, dtype=torch.float32, device=dev),
               src_token=torch.full((R, R, m), -7, dtype=torch.int32, device=dev),
               recv_counts=torch.full((R, R), -7, dtype=torch.int32, device=dev),
               local_expert_counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               recv_topk_ids=torch.full((R, R, m, K), -7, dtype=torch.int32, device=dev),
               recv_topk_w=torch.full((R, R, m, K), -7.0, dtype=torch.float32, device=dev),
               flags=torch.zeros((1,), dtype=torch.int32, device=dev))
    st = mod.moe_route_static_scratch(
        R, E, K, T, m, ids.data_ptr(), w.data_ptr(), out["send_slot"].data_ptr(),
        out["dest_weight"].data_ptr(), out["src_token"].data_ptr(),
        out["recv_counts"].data_ptr(), out["local_expert_counts"].data_ptr(),
        out["recv_topk_ids"].data_ptr(), out["recv_topk_w"].data_ptr(),
        out["flags"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == mod.MOE_OK, mod.status_string(st)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def dispatch_route(mod, R, E, K, T, m, H, ids, w):
    a2a = mod.MoeA2A(R, m, H, E, K, "cuda")
    x = torch.zeros((R, T, H), dtype=torch.bfloat16, device="cuda")
    v = a2a.dispatch(ids, w, x, m)
    torch.cuda.synchronize()
    ref = dict(send_slot=v.send_slot.cpu().numpy(), dest_weight=v.dest_weight.cpu().numpy(),
               src_token=v.src_token.cpu().numpy(), recv_counts=v.recv_counts.cpu().numpy(),
               local_expert_counts=v.local_expert_counts.cpu().numpy().ravel(),
               recv_topk_ids=v.recv_topk_ids.cpu().numpy(),
               recv_topk_w=v.recv_topk_w.cpu().numpy())
    a2a.combine(None, False)       # return the handle to idle
    return ref


def assert_same(got, ref, R):
    assert np.array_equal(got["recv_counts"], ref["recv_counts"])
    assert np.array_equal(got["local_expert_counts"], ref["local_expert_counts"])
    assert np.array_equal(got["send_slot"], ref["send_slot"])
    assert np.array_equal(got["dest_weight"].view(np.uint32), ref["dest_weight"].view(np.uint32))
    counts = ref["recv_counts"]
    for d in range(R):
        for s in range(R):
            c = counts[d, s]
            assert np.array_equal(got["src_token"][d, s, :c], ref["src_token"][d, s, :c])
            assert np.array_equal(got["recv_topk_ids"][d, s, :c], ref["recv_topk_ids"][d, s, :c])
            assert np.array_equal(got["recv_topk_w"][d, s, :c].view(np.uint32),
                                  ref["recv_topk_w"][d, s, :c].view(np.uint32))
    assert got["flags"][0] == 0


def test_static_scratch_matches_dispatch_on_consecutive_calls(mod):
    # two calls in a row on the shared array: a prefill-shaped Zipf routing,
    # then a smaller uniform one with a different top-k and plane stride
    calls = [(8, 256, 8, 4096, 4096, "zipf", 0), (6, 48, 5, 300, 310, "uniform", 1)]
    for R, E, K, T, m, routing, seed in calls:
        ids_h = synth.topk_ids(seed, R, T, E, K, routing)
        w_h = synth.topk_weights(seed, R, T, K)
        ids = torch.from_numpy(ids_h).cuda()
        w = torch.from_numpy(w_h).cuda()
        got = static_route(mod, R, E, K, T, m, ids, w)
        ref = dispatch_route(mod, R, E, K, T, m, 64, ids, w)
        assert_same(got, ref, R)


def test_static_scratch_rejects_sizes_beyond_its_array(mod):
    R, E, T = 32, 8192, 1 << 20
    assert mod.moe_route_static_scratch_bytes(R, E, T) > mod.MOE_STATIC_SCRATCH_BYTES
    dummy = 1 << 20                 # never touched: the size check comes first
    st = mod.moe_route_static_scratch(R, E, 8, T, T, *([dummy] * 9))
    assert st == mod.MOE_ERR_CAPACITY
