"""The allocation-free routing entry point, checked against the oracle and
against moe_dispatch.

moe_route_static_scratch serves callers that cannot allocate device memory
(a plugin inside a framework that owns the memory pool, a serving loop that
forbids cudaMalloc after start-up): they pass inputs and outputs, and the
routing pass's temporary memory is the library's fixed device array.  Its
outputs must equal the CPU oracle's routing, and the ones moe_dispatch
produces for the same routing, bit for bit, on consecutive calls that reuse
the shared array.  This file is collected last on purpose.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from combine_topk_ids_rank_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from oracle import oracle  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mod():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()
    from combine_topk_ids_rank_gb300 import moe_a2a
    return moe_a2a


def static_route(mod, R, E, K, T, m, ids, w, with_flags=True):
    RP = (R + 3) // 4 * 4
    dev = "cuda"
    out = dict(send_slot=torch.full((R, T, RP), -7, dtype=torch.int32, device=dev),
               dest_weight=torch.full((R, T, RP), -7.0, dtype=torch.float32, device=dev),
               src_token=torch.full((R, R, m), -7, dtype=torch.int32, device=dev),
               recv_counts=torch.full((R, R), -7, dtype=torch.int32, device=dev),
               local_expert_counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               recv_topk_ids=torch.full((R, R, m, K), -7, dtype=torch.int32, device=dev),
               recv_topk_w=torch.full((R, R, m, K), -7.0, dtype=torch.float32, device=dev),
               flags=torch.zeros((1,), dtype=torch.int32, device=dev))
    ptr = (lambda t: t.data_ptr() if t is not None and t.numel() else 0)
    st = mod.moe_route_static_scratch(
        R, E, K, T, m, ptr(ids), ptr(w), ptr(out["send_slot"]),
        ptr(out["dest_weight"]), ptr(out["src_token"]),
        out["recv_counts"].data_ptr(), out["local_expert_counts"].data_ptr(),
        ptr(out["recv_topk_ids"]), ptr(out["recv_topk_w"]),
        out["flags"].data_ptr() if with_flags else 0,
        torch.cuda.current_stream().cuda_stream)
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


def oracle_route(R, E, K, T, m, ids_h, w_h):
    """The oracle's routing tables and metadata rows, in the layout of the
    entry point's outputs (send rows padded to RP, padding entries -1 / 0)."""
    RP = (R + 3) // 4 * 4
    r = oracle.route(ids_h, w_h, E, m)
    od = oracle.dispatch(ids_h, w_h, np.zeros((R, T, 8), np.uint16), E, m, r)
    ss = np.full((R, T, RP), -1, np.int32)
    ss[:, :, :R] = r["send_slot"]
    dw = np.zeros((R, T, RP), np.float32)
    dw[:, :, :R] = r["wd"]
    return dict(send_slot=ss, dest_weight=dw, src_token=r["src_token"],
                recv_counts=r["recv_counts"],
                local_expert_counts=r["local_expert_counts"].ravel(),
                recv_topk_ids=od["recv_ids"], recv_topk_w=od["recv_w"],
                invalid=r["invalid"])


def assert_same(got, ref, R, T):
    assert np.array_equal(got["recv_counts"], ref["recv_counts"])
    assert np.array_equal(got["local_expert_counts"], ref["local_expert_counts"])
    assert np.array_equal(got["send_slot"][:, :T, :R], ref["send_slot"][:, :T, :R])
    assert np.array_equal(got["dest_weight"][:, :T, :R].view(np.uint32),
                          ref["dest_weight"][:, :T, :R].view(np.uint32))
    counts = ref["recv_counts"]
    for d in range(R):
        for s in range(R):
            c = counts[d, s]
            assert np.array_equal(got["src_token"][d, s, :c], ref["src_token"][d, s, :c])
            assert np.array_equal(got["recv_topk_ids"][d, s, :c], ref["recv_topk_ids"][d, s, :c])
            assert np.array_equal(got["recv_topk_w"][d, s, :c].view(np.uint32),
                                  ref["recv_topk_w"][d, s, :c].view(np.uint32))
            # slots past a count are never written (they keep the fill)
            assert (got["src_token"][d, s, c:] == -7).all()


def test_static_scratch_matches_oracle_and_dispatch_on_consecutive_calls(mod):
    # two calls in a row on the shared array: a prefill-shaped Zipf routing,
    # then a smaller uniform one with a different top-k and plane stride
    calls = [(8, 256, 8, 4096, 4096, "zipf", 0), (6, 48, 5, 300, 310, "uniform", 1)]
    for R, E, K, T, m, routing, seed in calls:
        ids_h = synth.topk_ids(seed, R, T, E, K, routing)
        w_h = synth.topk_weights(seed, R, T, K)
        ids = torch.from_numpy(ids_h).cuda()
        w = torch.from_numpy(w_h).cuda()
        got = static_route(mod, R, E, K, T, m, ids, w)
        assert got["flags"][0] == 0
        assert_same(got, oracle_route(R, E, K, T, m, ids_h, w_h), R, T)
        assert_same(got, dispatch_route(mod, R, E, K, T, m, 64, ids, w), R, T)


def test_static_scratch_empty_call_zeroes_the_counts(mod):
    # T = 0 after a call that left nonzero counts: recv_counts and
    # local_expert_counts come back zero, nothing else is needed
    got = static_route(mod, 4, 32, 4, 0, 8, None, None)
    assert (got["recv_counts"] == 0).all() and (got["local_expert_counts"] == 0).all()
    assert got["flags"][0] == 0


def test_static_scratch_without_a_flag_buffer_and_with_bad_ids(mod):
    R, E, K, T, m = 4, 16, 4, 300, 300
    ids_h = synth.topk_ids(2, R, T, E, K, "uniform")
    w_h = synth.topk_weights(2, R, T, K)
    ids = torch.from_numpy(ids_h).cuda()
    w = torch.from_numpy(w_h).cuda()
    # no flag output: the flags go to the array's own sink word
    got = static_route(mod, R, E, K, T, m, ids, w, with_flags=False)
    assert_same(got, oracle_route(R, E, K, T, m, ids_h, w_h), R, T)
    # ids outside [-1, E) raise the flag, are skipped, and the rest is routed
    bad = ids_h.copy()
    bad[0, 3, 1] = E
    bad[2, 7, 0] = -5
    bad[1, 1, :] = -1                 # the sentinel is fine
    got = static_route(mod, R, E, K, T, m, torch.from_numpy(bad).cuda(), w)
    assert got["flags"][0] == mod.MOE_DEVICE_FLAG_BAD_EXPERT_ID
    ref = oracle_route(R, E, K, T, m, bad, w_h)
    assert ref["invalid"] == 2
    assert_same(got, ref, R, T)


def test_static_scratch_rejects_sizes_beyond_its_array(mod):
    R, E, T = 32, 8192, 1 << 20
    assert mod.moe_route_static_scratch_bytes(R, E, T) > mod.MOE_STATIC_SCRATCH_BYTES
    dummy = 1 << 20                 # never touched: the size check comes first
    st = mod.moe_route_static_scratch(R, E, 8, T, T, *([dummy] * 9))
    assert st == mod.MOE_ERR_CAPACITY


def test_static_scratch_set_up_is_refused_during_capture():
    # A fresh process: the first call in its context, made while the stream
    # is capturing, must queue nothing and return MOE_ERR_SETUP_IN_CAPTURE
    # (the address lookup is made outside capture only).
    code = textwrap.dedent("""
        import torch
        from combine_topk_ids_rank_gb300 import moe_a2a as mod
        R, E, K, T = 2, 8, 2, 4
        ids = torch.zeros((R, T, K), dtype=torch.int32, device="cuda")
        w = torch.zeros((R, T, K), dtype=torch.float32, device="cuda")
        outs = [torch.zeros(1 << 14, dtype=torch.int32, device="cuda") for _ in range(7)]
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.capture_begin()
            st = mod.moe_route_static_scratch(R, E, K, T, T, ids.data_ptr(), w.data_ptr(),
                                              *[o.data_ptr() for o in outs], 0, s.cuda_stream)
            g.capture_end()
        print("status", st)
    """)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    from combine_topk_ids_rank_gb300 import moe_a2a as mod
    assert ("status %d" % mod.MOE_ERR_SETUP_IN_CAPTURE) in r.stdout, r.stdout + r.stderr[-2000:]
