"""Contract of the C ABI on the GPU: phase errors, the device flag for bad
expert ids, empty input, tokens without experts, in-place residual, the
zero-copy payload region, exactly-once reduction, no leakage between calls.
"""
import numpy as np
import pytest

from combine_topk_ids_rank_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import parity  # noqa: E402
from oracle import oracle  # noqa: E402


@pytest.fixture(scope="module")
def mod():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()
    from combine_topk_ids_rank_gb300 import moe_a2a
    return moe_a2a


def dev(a, dt):
    return parity.to_dev(a, dt)


def make(mod, R=4, M=64, H=128, E=16, K=4):
    return mod.MoeA2A(R, M, H, E, K, "cuda")


def inputs(R=4, T=32, H=128, E=16, K=4, seed=0):
    return dict(topk_ids=synth.topk_ids(seed, R, T, E, K),
                topk_w=synth.topk_weights(seed, R, T, K),
                x=synth.per_rank_rows(seed, synth.X, R, T, H),
                residual=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                gamma=synth.gamma(seed, H))


def test_dispatch_twice_is_a_phase_error(mod):
    a = make(mod)
    i = inputs()
    args = (dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32),
            dev(i["x"], torch.bfloat16))
    a.dispatch(*args)
    with pytest.raises(mod.MoeA2AError) as e:
        a.dispatch(*args)
    assert e.value.status == mod.MOE_ERR_PHASE and a.phase == 1
    a.combine(a.last_view.recv_x)
    assert a.phase == 0
    with pytest.raises(mod.MoeA2AError) as e:
        a.combine(a.last_view.recv_x)       # state reset after combine
    assert e.value.status == mod.MOE_ERR_PHASE


def test_capacity_errors_on_device_handle(mod):
    a = make(mod, M=64)
    i = inputs(T=32)
    args = (dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32),
            dev(i["x"], torch.bfloat16))
    for m in (16, 65):
        with pytest.raises(mod.MoeA2AError) as e:
            a.dispatch(*args, runtime_max_tokens_per_rank=m)
        assert e.value.status == mod.MOE_ERR_CAPACITY
    assert a.phase == 0


def test_bad_expert_ids_raise_the_device_flag(mod):
    a = make(mod)
    i = inputs()
    ids = i["topk_ids"].copy()
    ids[0, 3, 1] = 16          # == E
    ids[2, 7, 0] = -5
    ids[1, 1, :] = -1          # the sentinel is fine
    view = a.dispatch(dev(ids, torch.int32), dev(i["topk_w"], torch.float32),
                      dev(i["x"], torch.bfloat16))
    st, flags = a.get_error()
    assert st == mod.MOE_ERR_ROUTING and flags == mod.MOE_DEVICE_FLAG_BAD_EXPERT_ID
    assert a.get_error() == (mod.MOE_OK, 0)          # read clears it
    r = oracle.route(ids, i["topk_w"], 16, 32)
    assert r["invalid"] == 2
    assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"])
    assert np.array_equal(view.send_slot.cpu().numpy()[:, :, :4], r["send_slot"])
    a.combine(view.recv_x)


def test_empty_input(mod):
    a = make(mod)
    e = torch.empty((4, 0, 4), dtype=torch.int32, device="cuda")
    view = a.dispatch(e, e.float(), torch.empty((4, 0, 128), dtype=torch.bfloat16,
                                                device="cuda"), runtime_max_tokens_per_rank=8)
    assert view.recv_counts.sum().item() == 0
    assert view.local_expert_counts.sum().item() == 0
    out = a.combine(None, True)
    assert out.shape == (4, 0, 128) and a.phase == 0
    assert a.get_error() == (mod.MOE_OK, 0)


def test_tokens_without_experts(mod):
    a = make(mod)
    i = inputs()
    ids = i["topk_ids"].copy()
    ids[:, ::3, :] = -1
    view = a.dispatch(dev(ids, torch.int32), dev(i["topk_w"], torch.float32),
                      dev(i["x"], torch.bfloat16))
    res = dev(i["residual"], torch.bfloat16)
    gam = dev(i["gamma"], torch.bfloat16)
    out = a.combine(view.recv_x, True, res, gam, 1e-6)
    r = oracle.route(ids, i["topk_w"], 16, 32)
    od = oracle.dispatch(ids, i["topk_w"], i["x"], 16, 32, r)
    oc = oracle.combine(r, od["recv_x"], True, i["residual"], i["gamma"], 1e-6)
    y = parity.f32(parity.to_host_u16(out)).reshape(-1, 128).astype(np.float64)
    assert np.all(np.abs(y - oc["y"]) <= 2e-2)
    # unfused: a token with no expert combines to exactly zero
    view = a.dispatch(dev(ids, torch.int32), dev(i["topk_w"], torch.float32),
                      dev(i["x"], torch.bfloat16))
    out = a.combine(view.recv_x, False)
    assert torch.count_nonzero(out[:, ::3].float()).item() == 0


def test_in_place_residual_and_external_expert_out(mod):
    R, T, H = 4, 32, 128
    i = inputs()
    outs = []
    for mode in ("payload", "external", "inplace"):
        a = make(mod)
        view = a.dispatch(dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32),
                          dev(i["x"], torch.bfloat16))
        counts = view.recv_counts.cpu().numpy()
        eo = synth.expert_out_planes(9, R, T, H, counts)
        eo_dev = torch.zeros((R, R, T, H), dtype=torch.bfloat16, device="cuda")
        for d in range(R):
            for s in range(R):
                eo_dev[d, s, :counts[d, s]] = dev(eo[d, s, :counts[d, s]], torch.bfloat16)
        res = dev(i["residual"], torch.bfloat16)
        gam = dev(i["gamma"], torch.bfloat16)
        if mode == "payload":
            a.combine_payload().copy_(eo_dev)
            rout = torch.empty_like(res)
            y = a.combine(None, True, res, gam, 1e-6, residual_out=rout)
        elif mode == "external":
            rout = torch.empty_like(res)
            y = a.combine(eo_dev, True, res, gam, 1e-6, residual_out=rout)
        else:
            y = a.combine(eo_dev, True, res, gam, 1e-6, residual_out=res)
            rout = res
        outs.append((parity.to_host_u16(y), parity.to_host_u16(rout)))
    for y, rout in outs[1:]:
        assert np.array_equal(y, outs[0][0]) and np.array_equal(rout, outs[0][1])


def test_weighted_identity_reduces_exactly_once(mod):
    # top-k weights 1/8 sum to exactly 1: the combine of identity experts is x
    # itself, bit for bit (a second reduction would give 2x)
    R, T, H, E, K = 8, 48, 7168, 256, 8
    a = mod.MoeA2A(R, T, H, E, K, "cuda")
    ids = synth.topk_ids(1, R, T, E, K)
    w = np.full((R, T, K), 1.0 / K, np.float32)
    x = synth.per_rank_rows(1, synth.X, R, T, H)
    view = a.dispatch(dev(ids, torch.int32), dev(w, torch.float32), dev(x, torch.bfloat16))
    out = a.combine(view.recv_x, True)
    assert np.array_equal(parity.to_host_u16(out), x)


def test_no_leakage_between_calls(mod):
    # a large call followed by a small one on the same handle gives the same
    # result as the small call on a fresh, poisoned handle
    from dataclasses import replace
    w = replace(synth.WORKLOADS["decode"], tokens_per_rank=64, max_tokens=64,
                runtime_max=64, hidden=512)
    shared = parity.Case(w)
    shared.run(T=64, seed=1)
    small = replace(w, tokens_per_rank=10, runtime_max=12)
    shared.w = small
    rep = shared.run(seed=2)
    assert rep["T"] == 10


@pytest.mark.parametrize("fp8", [False, True])
def test_handles_of_different_sizes_interleaved(mod, fp8):
    # Two handles with different hidden sizes in one process, the larger
    # prepared first: each kernel's shared-memory limit is one per process,
    # so preparing the smaller handle must not take it below what the larger
    # one launches with.  Both stay usable, and both match the oracle, on the
    # one-launch dispatch, the routing passes + row copy and the combines.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    R, E, K = 4, 16, 4
    handles = {}
    for H in (2048, 512):          # the larger first
        handles[H] = MoeA2A(R, 300, H, E, K, "cuda")
        if fp8:
            handles[H].set_recv_format(MOE_FORMAT_FP8_E4M3)
    for rnd in range(2):
        for H in (2048, 512):
            for T in (40, 300):    # one launch, then the routing passes
                a = handles[H]
                seed = 100 * rnd + T + H
                ids = synth.topk_ids(seed, R, T, E, K)
                w = synth.topk_weights(seed, R, T, K)
                x = synth.per_rank_rows(seed, synth.X, R, T, H)
                res = synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H)
                gam = synth.gamma(seed, H)
                view = a.dispatch(dev(ids, torch.int32), dev(w, torch.float32),
                                  dev(x, torch.bfloat16))
                r = oracle.route(ids, w, E, T)
                assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"])
                eo = synth.expert_out_planes(seed, R, T, H, r["recv_counts"])
                if fp8:
                    q_ref, s_ref = oracle.quantize_rows_fp8(x)
                    codes = view.recv_x.view(torch.uint8).cpu().numpy()
                    src = view.src_token.cpu().numpy()
                    for d in range(R):
                        for s in range(R):
                            for j in range(r["recv_counts"][d, s]):
                                assert np.array_equal(codes[d, s, j], q_ref[s, src[d, s, j]])
                    a.combine_payload().copy_(dev(eo, torch.bfloat16))
                    rout = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
                    out = a.combine(None, True, dev(res, torch.bfloat16),
                                    dev(gam, torch.bfloat16), 1e-6, residual_out=rout)
                else:
                    od = oracle.dispatch(ids, w, x, E, T, r)
                    rx = parity.to_host_u16(view.recv_x)
                    for d in range(R):
                        for s in range(R):
                            c = r["recv_counts"][d, s]
                            assert np.array_equal(rx[d, s, :c], od["recv_x"][d, s, :c])
                    eo = od["recv_x"]
                    rout = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
                    out = a.combine(view.recv_x, True, dev(res, torch.bfloat16),
                                    dev(gam, torch.bfloat16), 1e-6, residual_out=rout)
                torch.cuda.synchronize()
                assert a.get_error() == (mod.MOE_OK, 0)
                oc = oracle.combine(r, eo, True, res, gam, 1e-6)
                assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H),
                                      oc["residual_out"]), (H, T, rnd)
                y = parity.f32(parity.to_host_u16(out)).reshape(-1, H).astype(np.float64)
                err = np.abs(y - oc["y"])
                assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()


def test_dispatch_and_combine_on_two_user_streams(mod):
    # The inputs are written on stream 1 after a long sleep there; dispatch
    # runs on stream 1 (its second routing pass on the handle's own stream,
    # forked from and joined back into the caller's), and the combine on
    # stream 2 after stream 2 waits for stream 1 only.  Any step that ran on
    # another stream without those dependencies would read stale inputs or
    # tables; every result must be the oracle's.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    R, T, H, E, K = 4, 300, 256, 32, 4           # the routing passes (T > 256)
    a = MoeA2A(R, T, H, E, K, "cuda")
    i = inputs(seed=77, R=R, T=T, H=H, E=E, K=K)
    ids = torch.zeros((R, T, K), dtype=torch.int32, device="cuda")
    w = torch.zeros((R, T, K), dtype=torch.float32, device="cuda")
    x = torch.zeros((R, T, H), dtype=torch.bfloat16, device="cuda")
    ids_h, w_h, x_h = dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32), \
        dev(i["x"], torch.bfloat16)
    res, gam = dev(i["residual"], torch.bfloat16), dev(i["gamma"], torch.bfloat16)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for rnd in range(3):
        with torch.cuda.stream(s1):
            torch.cuda._sleep(20_000_000)          # ~10 ms of spinning on stream 1
            ids.copy_(ids_h)
            w.copy_(w_h)
            x.copy_(x_h)
            view = a.dispatch(ids, w, x)
        s2.wait_stream(s1)
        with torch.cuda.stream(s2):
            rout = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
            out = a.combine(view.recv_x, True, res, gam, 1e-6, residual_out=rout)
        torch.cuda.synchronize()
        assert a.get_error(s2) == (mod.MOE_OK, 0)
        r = oracle.route(i["topk_ids"], i["topk_w"], E, T)
        assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"]), rnd
        od = oracle.dispatch(i["topk_ids"], i["topk_w"], i["x"], E, T, r)
        oc = oracle.combine(r, od["recv_x"], True, i["residual"], i["gamma"], 1e-6)
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"]), rnd
        y = parity.f32(parity.to_host_u16(out)).reshape(-1, H).astype(np.float64)
        err = np.abs(y - oc["y"])
        assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all(), rnd
        ids.zero_(), w.zero_(), x.zero_()           # (on the current stream, after the sync)
        torch.cuda.synchronize()


def test_many_handles_created_and_destroyed(mod):
    # create, use and destroy handles repeatedly: every call succeeds, the
    # results stay the oracle's, and no device memory is left behind
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    R, T, H, E, K = 4, 40, 128, 16, 4
    i = inputs(seed=78, R=R, T=T, H=H, E=E, K=K)
    r = oracle.route(i["topk_ids"], i["topk_w"], E, T)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    for n in range(50):
        a = MoeA2A(R, T, H, E, K, "cuda")
        view = a.dispatch(dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32),
                          dev(i["x"], torch.bfloat16))
        out = a.combine(view.recv_x, False)
        if n % 10 == 0:
            torch.cuda.synchronize()
            assert a.get_error() == (mod.MOE_OK, 0)
            assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"])
        a.close()
        del a, view, out
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == base


def test_two_host_threads_with_their_own_handles(mod):
    # Distinct handles are independent: two host threads, each with its own
    # handle (different sizes, so each prepares its own kernel shapes while
    # the other runs) and its own stream, dispatch and combine at the same
    # time; every call's result is the oracle's.
    import threading
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    cfgs = [dict(R=4, T=300, H=512, E=16, K=4, seed=81), dict(R=8, T=40, H=2048, E=64, K=8, seed=82)]
    expect, inputs_dev = [], []
    for c in cfgs:
        i = inputs(seed=c["seed"], R=c["R"], T=c["T"], H=c["H"], E=c["E"], K=c["K"])
        r = oracle.route(i["topk_ids"], i["topk_w"], c["E"], c["T"])
        od = oracle.dispatch(i["topk_ids"], i["topk_w"], i["x"], c["E"], c["T"], r)
        oc = oracle.combine(r, od["recv_x"], True, i["residual"], i["gamma"], 1e-6)
        expect.append((r, oc))
        inputs_dev.append([dev(i["topk_ids"], torch.int32), dev(i["topk_w"], torch.float32),
                           dev(i["x"], torch.bfloat16), dev(i["residual"], torch.bfloat16),
                           dev(i["gamma"], torch.bfloat16)])
    torch.cuda.synchronize()
    errors = []
    barrier = threading.Barrier(len(cfgs))

    def work(k):
        try:
            c, (r, oc) = cfgs[k], expect[k]
            ids, w, x, res, gam = inputs_dev[k]
            stream = torch.cuda.Stream()
            barrier.wait()
            a = MoeA2A(c["R"], c["T"], c["H"], c["E"], c["K"], "cuda")
            with torch.cuda.stream(stream):
                for _ in range(20):
                    view = a.dispatch(ids, w, x)
                    rout = torch.empty_like(res)
                    out = a.combine(view.recv_x, True, res, gam, 1e-6, residual_out=rout)
                stream.synchronize()
            assert a.get_error(stream) == (mod.MOE_OK, 0)
            assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"])
            H = c["H"]
            assert np.array_equal(parity.to_host_u16(rout).reshape(-1, H), oc["residual_out"])
            y = parity.f32(parity.to_host_u16(out)).reshape(-1, H).astype(np.float64)
            err = np.abs(y - oc["y"])
            assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()
            a.close()
        except Exception as e:          # reported by the main thread
            errors.append((k, repr(e)))

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(cfgs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
