"""CUDA-graph capture of a dispatch + combine pair, replayed on new inputs.

The inputs live in fixed device buffers; each replay follows a copy of a new
seeded input set into them, and every replay's routing, counts (the
local-expert counts included), dispatched rows and combine outputs must be
the oracle's for that input set.  The experts are the identity (the combine
reads the dispatched rows), so the whole pair runs on the device.  A batch
that a direct call dispatches in one launch is captured through the routing
passes, whose accumulators are cleared inside each call.
"""
from dataclasses import replace

import numpy as np
import pytest

from combine_topk_ids_rank_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import parity  # noqa: E402
from oracle import oracle  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()


@pytest.mark.parametrize("T", [40, 300])
def test_graph_replays_match_the_oracle(T):
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    R, M, H, E, K = 4, 300, 256, 32, 4
    w = replace(synth.WORKLOADS["decode"], ep_size=R, tokens_per_rank=T, max_tokens=M,
                runtime_max=T, hidden=H, num_experts=E, top_k=K, weighted=True, fused=True)
    a = MoeA2A(R, M, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)

    def inputs(seed):
        inp = synth.inputs(w, seed)
        return {k: np.ascontiguousarray(inp[k]) for k in ("topk_ids", "topk_w", "x", "residual",
                                                          "gamma")}

    first = inputs(100)
    ids = parity.to_dev(first["topk_ids"], torch.int32)
    wts = parity.to_dev(first["topk_w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    res = parity.to_dev(first["residual"], torch.bfloat16)
    gam = parity.to_dev(first["gamma"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(res)

    # a direct call first (it also creates the handle's stream and events)
    view = a.dispatch(ids, wts, x, T)
    assert view.kernels == (1 if T <= 256 else 3)
    a.combine(view.recv_x, True, res, gam, w.eps, out, rout)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = a.dispatch(ids, wts, x, T)
        a.combine(view.recv_x, True, res, gam, w.eps, out, rout)
    assert view.kernels == 3  # captured through the routing passes
    assert a.phase == 0

    for seed in (1, 2, 3):
        inp = inputs(seed)
        ids.copy_(parity.to_dev(inp["topk_ids"], torch.int32))
        wts.copy_(parity.to_dev(inp["topk_w"], torch.float32))
        x.copy_(parity.to_dev(inp["x"], torch.bfloat16))
        res.copy_(parity.to_dev(inp["residual"], torch.bfloat16))
        gam.copy_(parity.to_dev(inp["gamma"], torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        st, flags = a.get_error()
        assert st == 0 and flags == 0, (st, flags)

        r = oracle.route(inp["topk_ids"], inp["topk_w"], E, T)
        counts = view.recv_counts.cpu().numpy()
        assert np.array_equal(counts, r["recv_counts"]), ("recv_counts", seed)
        assert np.array_equal(view.local_expert_counts.cpu().numpy(),
                              r["local_expert_counts"]), ("local_expert_counts", seed)
        assert np.array_equal(view.send_slot.cpu().numpy()[:, :, :R], r["send_slot"]), seed
        od = oracle.dispatch(inp["topk_ids"], inp["topk_w"], inp["x"], E, T, r)
        gx = parity.to_host_u16(view.recv_x)
        for d in range(R):
            for s in range(R):
                c = counts[d, s]
                assert np.array_equal(gx[d, s, :c], od["recv_x"][d, s, :c]), (d, s, seed)

        oc = oracle.combine(r, od["recv_x"], True, inp["residual"], inp["gamma"], w.eps,
                            tokens=np.arange(R * T))
        g_rout = parity.to_host_u16(rout).reshape(R * T, H)
        assert np.array_equal(g_rout, oc["residual_out"]), ("residual_out", seed)
        y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
        err = np.abs(y - oc["y"])
        bad = (err > parity.ABS_TOL) | (err > parity.REL_TOL * np.abs(oc["y"]))
        assert not bad.any(), ("RMSNorm tolerance", seed, float(err.max()))


def test_graph_replays_expert_layout():
    # The expert-major layout (one row per (token, expert), the gates applied
    # in the combine): its two routing passes move the expert histogram out of
    # an accumulator and clear it inside each call, so replays stay exact.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_LAYOUT_EXPERT
    R, T, H, E, K = 4, 50, 128, 16, 4
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)

    def inputs(seed):
        return dict(ids=synth.topk_ids(seed, R, T, E, K, "uniform"),
                    w=synth.topk_weights(seed, R, T, K),
                    x=synth.per_rank_rows(seed, synth.X, R, T, H),
                    res=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                    g=synth.gamma(seed, H))

    first = inputs(200)
    ids = parity.to_dev(first["ids"], torch.int32)
    wts = parity.to_dev(first["w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    res = parity.to_dev(first["res"], torch.bfloat16)
    gam = parity.to_dev(first["g"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(res)
    view = a.dispatch(ids, wts, x, T)
    a.combine(view.recv_x, True, res, gam, 1e-6, out, rout)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = a.dispatch(ids, wts, x, T)
        a.combine(view.recv_x, True, res, gam, 1e-6, out, rout)

    for seed in (4, 5, 6):
        inp = inputs(seed)
        for dst, src, dt in ((ids, inp["ids"], torch.int32), (wts, inp["w"], torch.float32),
                             (x, inp["x"], torch.bfloat16), (res, inp["res"], torch.bfloat16),
                             (gam, inp["g"], torch.bfloat16)):
            dst.copy_(parity.to_dev(src, dt))
        g.replay()
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        r = oracle.route_experts(inp["ids"], inp["w"], E, T)
        assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"]), seed
        assert np.array_equal(view.local_expert_counts.cpu().numpy(),
                              r["local_expert_counts"]), seed
        rx = oracle.dispatch_experts(inp["x"], E, T, r)
        oc = oracle.combine_experts(r, rx, True, inp["res"], inp["g"], 1e-6,
                                    tokens=np.arange(R * T))
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H),
                              oc["residual_out"]), ("residual_out", seed)
        y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
        err = np.abs(y - oc["y"])
        assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"])).all()


def test_graph_replays_fp8_dispatch():
    # FP8 receive rows: every replay's e4m3 codes and per-row scales are the
    # oracle's quantisation of that replay's rows; the combine (bf16 output)
    # reads a payload written once, at the slots of each replay's routing.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    R, T, H, E, K = 4, 30, 256, 32, 4
    w = replace(synth.WORKLOADS["decode"], ep_size=R, tokens_per_rank=T, max_tokens=T,
                runtime_max=T, hidden=H, num_experts=E, top_k=K, weighted=True, fused=False)
    a = MoeA2A(R, T, H, E, K, "cuda")
    a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    first = synth.inputs(w, 300)
    ids = parity.to_dev(first["topk_ids"], torch.int32)
    wts = parity.to_dev(first["topk_w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    view = a.dispatch(ids, wts, x, T)
    eo = synth.expert_out_planes(7, R, T, H, np.full((R, R), T))  # every slot drawn
    a.combine_payload().copy_(parity.to_dev(eo, torch.bfloat16))
    a.combine(None, True, out=out)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = a.dispatch(ids, wts, x, T)
        a.combine(None, True, out=out)

    for seed in (7, 8, 9):
        inp = synth.inputs(w, seed)
        ids.copy_(parity.to_dev(inp["topk_ids"], torch.int32))
        wts.copy_(parity.to_dev(inp["topk_w"], torch.float32))
        x.copy_(parity.to_dev(inp["x"], torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        r = oracle.route(inp["topk_ids"], inp["topk_w"], E, T)
        counts = view.recv_counts.cpu().numpy()
        assert np.array_equal(counts, r["recv_counts"]), seed
        assert np.array_equal(view.local_expert_counts.cpu().numpy(),
                              r["local_expert_counts"]), seed
        q_ref, s_ref = oracle.quantize_rows_fp8(inp["x"])
        codes = view.recv_x.view(torch.uint8).cpu().numpy()
        scales = view.recv_scale.cpu().numpy()
        src = view.src_token.cpu().numpy()
        for d in range(R):
            for s in range(R):
                for j in range(counts[d, s]):
                    t = src[d, s, j]
                    assert np.array_equal(codes[d, s, j], q_ref[s, t]), (d, s, j, seed)
                    assert scales[d, s, j] == s_ref[s, t]
        oc = oracle.combine(r, eo, True, tokens=np.arange(R * T))
        assert np.array_equal(parity.to_host_u16(out).reshape(R * T, H), oc["out"]), seed


@pytest.mark.parametrize("fp8", [False, True])
def test_graph_replays_rank_plane_moe_step(fp8):
    # A whole MoE step on the rank planes captured once: dispatch, the
    # expert product with the gates (pair lists cleared inside each call),
    # the unweighted fused combine.  W_e = 2^(e mod 3) I (bf16, or unit
    # codes with that channel scale) makes each expert output exact, so the
    # gated sums are the same IEEE operations on both sides: the messages
    # equal the oracle's bit for bit on every replay.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    R, T, H, E, K = 4, 40, 256, 16, 4
    a = MoeA2A(R, T, H, E, K, "cuda")
    if fp8:
        a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    scale = (2.0 ** (np.arange(E) % 3)).astype(np.float32)
    if fp8:
        eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
        qw = np.ascontiguousarray(np.broadcast_to(eye, (E, H, H)))
        sw = np.repeat(scale[:, None], H, axis=1)
        qw_d, sw_d = parity.to_dev(qw, torch.uint8), parity.to_dev(sw, torch.float32)
        product = lambda: a.expert_gemm_rank_fp8(qw_d, sw_d, True)
    else:
        wb = parity.f32_to_bits(np.stack([np.eye(H, dtype=np.float32) * scale[e]
                                          for e in range(E)]))
        wb_d = parity.to_dev(wb, torch.bfloat16)
        product = lambda: a.expert_gemm_rank(wb_d, True)

    def inputs(seed):
        return dict(ids=synth.topk_ids(seed, R, T, E, K, "uniform"),
                    w=synth.topk_weights(seed, R, T, K),
                    x=synth.per_rank_rows(seed, synth.X, R, T, H),
                    res=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                    g=synth.gamma(seed, H))

    first = inputs(400)
    ids = parity.to_dev(first["ids"], torch.int32)
    wts = parity.to_dev(first["w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    res = parity.to_dev(first["res"], torch.bfloat16)
    gam = parity.to_dev(first["g"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(res)
    view = a.dispatch(ids, wts, x, T)          # direct calls first: stream, events, scratch
    product()
    a.combine(None, False, res, gam, 1e-6, out, rout)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = a.dispatch(ids, wts, x, T)
        product()
        a.combine(None, False, res, gam, 1e-6, out, rout)

    for seed in (41, 42, 43):
        inp = inputs(seed)
        for dst, src, dt in ((ids, inp["ids"], torch.int32), (wts, inp["w"], torch.float32),
                             (x, inp["x"], torch.bfloat16), (res, inp["res"], torch.bfloat16),
                             (gam, inp["g"], torch.bfloat16)):
            dst.copy_(parity.to_dev(src, dt))
        g.replay()
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        r = oracle.route(inp["ids"], inp["w"], E, T)
        counts = view.recv_counts.cpu().numpy()
        assert np.array_equal(counts, r["recv_counts"]), seed
        od = oracle.dispatch(inp["ids"], inp["w"], inp["x"], E, T, r)
        if fp8:
            q, sc = oracle.quantize_rows_fp8(inp["x"])
            qx = np.zeros((R, R, T, H), np.uint8)
            sx = np.zeros((R, R, T), np.float32)
            for d in range(R):
                for s in range(R):
                    c = counts[d, s]
                    qx[d, s, :c] = q[s, r["src_token"][d, s, :c]]
                    sx[d, s, :c] = sc[s, r["src_token"][d, s, :c]]
            msg = oracle.expert_gemm_rank_fp8(qx, sx, od["recv_ids"], od["recv_w"],
                                              r["recv_counts"], qw, sw, True)
        else:
            msg = oracle.expert_gemm_rank(od["recv_x"], od["recv_ids"], od["recv_w"],
                                          r["recv_counts"], wb, True)
        pay = parity.to_host_u16(a.combine_payload())
        for d in range(R):
            for s in range(R):
                c = counts[d, s]
                assert np.array_equal(pay[d, s, :c], msg[d, s, :c]), (d, s, seed)
        oc = oracle.combine(r, msg, False, inp["res"], inp["g"], 1e-6, tokens=np.arange(R * T))
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H),
                              oc["residual_out"]), ("residual_out", seed)
        y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
        err = np.abs(y - oc["y"])
        assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"])).all()


@pytest.mark.parametrize("mode", ["out8-fused", "tree", "varlen-dead"])
def test_graph_replays_combine_modes(mode):
    # Dispatch + combine captured once in the FP8-output, bf16-tree or
    # per-rank-count (with a dead rank) mode, replayed on three new input
    # sets (counts and the dead rank are host-side and fixed by the capture):
    # every replay equals the oracle on that replay's inputs.
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_REDUCE_BF16_TOPK_TREE
    R, T, H, E, K = 4, 60, 256, 32, 4
    counts = [60, 0, 33, 7]
    dead = 2
    a = MoeA2A(R, T, H, E, K, "cuda")
    if mode == "tree":
        a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
    if mode == "varlen-dead":
        a.set_active_ranks(0xF & ~(1 << dead))

    def inputs(seed):
        return dict(ids=synth.topk_ids(seed, R, T, E, K), w=synth.topk_weights(seed, R, T, K),
                    x=synth.per_rank_rows(seed, synth.X, R, T, H),
                    res=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                    g=synth.gamma(seed, H))

    first = inputs(500)
    ids = parity.to_dev(first["ids"], torch.int32)
    wts = parity.to_dev(first["w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    res = parity.to_dev(first["res"], torch.bfloat16)
    gam = parity.to_dev(first["g"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    out8 = torch.empty((R, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    osc = torch.empty((R, T), dtype=torch.float32, device="cuda")
    rout = torch.empty_like(res)

    def step():
        v = a.dispatch_varlen(ids, wts, x, counts) if mode == "varlen-dead" else \
            a.dispatch(ids, wts, x, T)
        if mode == "out8-fused":
            a.combine_fp8(v.recv_x, True, res, gam, 1e-6, out8, osc, rout)
        elif mode == "tree":
            a.combine(v.recv_x, False, out=out)
        else:
            a.combine(v.recv_x, True, res, gam, 1e-6, out, rout)
        return v

    view = step()                                  # direct first (stream, events)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = step()

    for seed in (51, 52, 53):
        inp = inputs(seed)
        for dst, src, dt in ((ids, inp["ids"], torch.int32), (wts, inp["w"], torch.float32),
                             (x, inp["x"], torch.bfloat16), (res, inp["res"], torch.bfloat16),
                             (gam, inp["g"], torch.bfloat16)):
            dst.copy_(parity.to_dev(src, dt))
        g.replay()
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        ids_o = inp["ids"].copy()
        live = np.ones((R, T), bool)
        if mode == "varlen-dead":
            for s, n in enumerate(counts):
                ids_o[s, n:] = -1
                live[s, n:] = False
            ids_o[(ids_o >= 0) & (ids_o // (E // R) == dead)] = -1
        tok = np.flatnonzero(live.ravel())
        r = oracle.route(ids_o, inp["w"], E, T)
        assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"]), (mode, seed)
        od = oracle.dispatch(ids_o, inp["w"], inp["x"], E, T, r)
        if mode == "tree":
            oc = oracle.combine_topk_tree(r, ids_o, E, od["recv_x"], tokens=tok)
            assert np.array_equal(parity.to_host_u16(out).reshape(R * T, H)[tok], oc["out"]), seed
            continue
        oc = oracle.combine(r, od["recv_x"], True, inp["res"], inp["g"], 1e-6, tokens=tok)
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H)[tok],
                              oc["residual_out"]), (mode, seed)
        y = oc["y"]
        if mode == "out8-fused":
            g_q = out8.view(torch.uint8).cpu().numpy().reshape(R * T, H)[tok]
            g_s = osc.cpu().numpy().ravel()[tok].astype(np.float64)
            deq = oracle.fp8_to_f32(g_q).astype(np.float64) * g_s[:, None]
            bound = (2.0 ** -4 + 1e-4) * np.abs(y) + 2.0 ** -10 * g_s[:, None] + 1e-6
            assert (np.abs(deq - y) <= bound).all(), seed
        else:
            got = parity.f32(parity.to_host_u16(out).reshape(R * T, H)[tok]).astype(np.float64)
            err = np.abs(got - y)
            assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(y))).all(), seed


@pytest.mark.parametrize("fp8", [False, True])
def test_graph_replays_expert_layout_moe_step(fp8):
    # A whole MoE step on the expert-major layout captured once: dispatch,
    # the expert product into the combine payload (it reads the rows per
    # expert of the current dispatch), the weighted fused combine.  Direct
    # calls first take the one-launch dispatch, which alternates its count
    # buffers; the captured call takes the routing passes.  W_e = 2^(e mod 3) I
    # (bf16, or unit codes with that channel scale) makes every expert output
    # exact, so each replay's outputs are the oracle's.
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MOE_LAYOUT_EXPERT,
                                                     MOE_FORMAT_FP8_E4M3)
    R, T, H, E, K = 4, 40, 256, 16, 4
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    if fp8:
        a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    scale = (2.0 ** (np.arange(E) % 3)).astype(np.float32)
    if fp8:
        eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
        qw_d = parity.to_dev(np.ascontiguousarray(np.broadcast_to(eye, (E, H, H))), torch.uint8)
        sw_d = parity.to_dev(np.repeat(scale[:, None], H, axis=1), torch.float32)
        product = lambda: a.expert_gemm_fp8(qw_d, sw_d)
    else:
        wb = parity.f32_to_bits(np.stack([np.eye(H, dtype=np.float32) * scale[e]
                                          for e in range(E)]))
        wb_d = parity.to_dev(wb, torch.bfloat16)
        product = lambda: a.expert_gemm(wb_d)

    def inputs(seed):
        return dict(ids=synth.topk_ids(seed, R, T, E, K), w=synth.topk_weights(seed, R, T, K),
                    x=synth.per_rank_rows(seed, synth.X, R, T, H),
                    res=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                    g=synth.gamma(seed, H))

    first = inputs(600)
    ids = parity.to_dev(first["ids"], torch.int32)
    wts = parity.to_dev(first["w"], torch.float32)
    x = parity.to_dev(first["x"], torch.bfloat16)
    res = parity.to_dev(first["res"], torch.bfloat16)
    gam = parity.to_dev(first["g"], torch.bfloat16)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(res)

    def step():
        v = a.dispatch(ids, wts, x, T)
        product()
        a.combine(None, True, res, gam, 1e-6, out, rout)
        return v

    for _ in range(3):                             # direct calls: the one-launch dispatch
        view = step()
        assert view.kernels == 1
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        view = step()
    assert view.kernels == 3

    for seed in (61, 62, 63):
        inp = inputs(seed)
        for dst, src, dt in ((ids, inp["ids"], torch.int32), (wts, inp["w"], torch.float32),
                             (x, inp["x"], torch.bfloat16), (res, inp["res"], torch.bfloat16),
                             (gam, inp["g"], torch.bfloat16)):
            dst.copy_(parity.to_dev(src, dt))
        g.replay()
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        r = oracle.route_experts(inp["ids"], inp["w"], E, T)
        cnt = view.recv_counts.cpu().numpy()
        assert np.array_equal(cnt, r["recv_counts"]), seed
        rx = oracle.dispatch_experts(inp["x"], E, T, r)
        cap = R * T
        eo = np.zeros((E, cap, H), np.uint16)
        if fp8:
            # the product's epilogue: bf16 of (f(qx) * sx) * sw, each product
            # rounded to binary32 (the sum is a single exact term)
            q, sc = oracle.quantize_rows_fp8(inp["x"])
            fq = oracle.fp8_to_f32(q).astype(np.float32)
            where, vals = [], []
            for e in range(E):
                for j in range(cnt[e]):
                    s, t = divmod(int(r["src_row"][e, j]), T)
                    where.append((e, j))
                    vals.append((fq[s, t] * np.float32(sc[s, t])) * np.float32(scale[e]))
            bits = oracle.bf16_bits(np.stack(vals)).reshape(len(vals), H)
            for (e, j), b in zip(where, bits):
                eo[e, j] = b
        else:
            for e in range(E):
                c = cnt[e]
                eo[e, :c] = parity.f32_to_bits(parity.f32(rx[e, :c]) * scale[e])
        oc = oracle.combine_experts(r, eo, True, inp["res"], inp["g"], 1e-6)
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"]), seed
        y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
        err = np.abs(y - oc["y"])
        assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all(), seed
