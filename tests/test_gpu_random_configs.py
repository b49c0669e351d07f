"""Seeded random configurations through dispatch and combine, against the oracle.

Each case draws a shape the fixed tests do not pin down: ranks 1-32 (not
only powers of two), 1-8 experts per rank, top-1 to top-8, hidden sizes from
one 16-byte vector to 7168 (ragged against a warp's vector span), batches on
either side of the one-launch dispatch's limit, a runtime maximum above the
batch, uniform or Zipf routing, weighted or not, fused or not; on the rank
layout with bf16 or FP8 rows, and on the expert layout.  Two more sweeps
draw shapes of the expert products (both layouts, bf16 and e4m3) and of the
combine modes (per-rank token counts with dead ranks, the bf16 top-k-slot
tree, the FP8 output).  The checks are the fixed tests' own (routing
tables, counts, rows or codes and scales, padding left untouched, combine
outputs), so a failure names its case by index and the drawn shape.
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

N_CASES = 96
FAMILIES = ("rank-bf16", "rank-fp8", "expert-bf16", "expert-fp8")
WORKSPACE_BUDGET = 1 << 30   # bytes of the two row regions of one case


def draw(i):
    """The i-th case: family and shape, from a generator seeded by i."""
    rng = np.random.default_rng(1000 + i)
    family = FAMILIES[i % len(FAMILIES)]
    fp8 = family.endswith("fp8")
    R = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 32]))
    Epr = int(rng.integers(1, 9))
    E = R * Epr
    K = int(rng.integers(1, min(8, E) + 1))
    H = int(rng.choice([16, 48, 64, 144, 512, 1040, 2048, 4112, 7168] if fp8 else
                       [8, 24, 64, 136, 512, 1032, 2048, 4104, 7168]))
    M = int(rng.choice([1, 7, 33, 64, 100, 256, 257, 300, 700]))
    planes = E * R if family.startswith("expert") else R * R
    while planes * M * H * 4 > WORKSPACE_BUDGET and M > 1:
        M = max(1, M // 2)
    T = int(rng.integers(0, M + 1))
    m = int(rng.integers(max(T, 1), M + 1))
    return dict(family=family, R=R, E=E, K=K, H=H, M=M, T=T, m=m,
                routing=str(rng.choice(["uniform", "zipf"])),
                weighted=bool(rng.integers(2)), fused=bool(rng.integers(2)), seed=i)


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()


def run_rank_bf16(c):
    w = replace(synth.WORKLOADS["tiny"], name="random", ep_size=c["R"], tokens_per_rank=c["T"],
                max_tokens=c["M"], runtime_max=c["m"], hidden=c["H"], num_experts=c["E"],
                top_k=c["K"], routing=c["routing"], weighted=c["weighted"], fused=c["fused"],
                identity_experts=False)
    case = parity.Case(w)
    rep = case.run(seed=c["seed"], sample=None)
    assert rep["T"] == c["T"]
    case.a2a.close()


def run_rank_fp8(c):
    import test_gpu_fp8 as f
    R, T, H, E, K, m = c["R"], c["T"], c["H"], c["E"], c["K"], c["m"]
    a, view, d = f.run_dispatch_fp8(R, T, H, E, K, c["seed"], m=m, routing=c["routing"])
    # combine of bf16 messages written into the payload, plain or fused
    cnt, r = d["cnt"], d["r"]
    eo = synth.expert_out_planes(c["seed"], R, m, H, cnt)
    pay = a.combine_payload()
    for dd in range(R):
        for s in range(R):
            if cnt[dd, s]:
                pay[dd, s, :cnt[dd, s]].copy_(parity.to_dev(eo[dd, s, :cnt[dd, s]], torch.bfloat16))
    res = synth.per_rank_rows(c["seed"], synth.RESIDUAL, R, T, H)
    gam = synth.gamma(c["seed"], H)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    if c["fused"]:
        rout = torch.empty_like(out)
        a.combine(None, c["weighted"], parity.to_dev(res, torch.bfloat16),
                  parity.to_dev(gam, torch.bfloat16), 1e-6, out, rout)
    else:
        a.combine(None, c["weighted"], out=out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 0
    oc = oracle.combine(r, eo, c["weighted"], res if c["fused"] else None,
                        gam if c["fused"] else None, 1e-6)
    got = parity.to_host_u16(out).reshape(R * T, H)
    if c["fused"]:
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"])
        y = parity.f32(got).astype(np.float64)
        err = np.abs(y - oc["y"])
        assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()
    else:
        assert np.array_equal(got, oc["out"])
    a.close()


def run_expert(c, fp8):
    import test_gpu_expert_layout as x
    x.run(c["R"], c["T"], c["H"], c["E"], c["K"], c["seed"], c["weighted"], c["fused"],
          m=c["m"], routing=c["routing"], fp8=fp8)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    c = draw(i)
    try:
        if c["family"] == "rank-bf16":
            run_rank_bf16(c)
        elif c["family"] == "rank-fp8":
            run_rank_fp8(c)
        else:
            run_expert(c, c["family"] == "expert-fp8")
    except AssertionError as e:
        raise AssertionError("case %d %s: %s" % (i, c, e)) from e


# --------------------------------------------------------------------------
# The expert-side products on random shapes: both layouts, bf16 or e4m3
# operands, experts that receive no row or a few (partial row tiles), one or
# several column tiles of 128 or 256.
# --------------------------------------------------------------------------

N_PRODUCT_CASES = 24


def draw_product(i):
    rng = np.random.default_rng(5000 + i)
    layout = ("rank", "expert")[i % 2]
    fp8 = bool((i // 2) % 2)
    R = int(rng.choice([1, 2, 3, 4, 8]))
    Epr = int(rng.integers(1, 5))
    E = R * Epr
    K = int(rng.integers(1, min(4, E) + 1))
    H = int(rng.choice([128, 256, 384, 640]))          # multiples of 128 (e4m3 stage rows)
    N = int(rng.choice([128, 256, 384, 512]))
    T = int(rng.integers(1, 161))
    return dict(layout=layout, fp8=fp8, R=R, E=E, K=K, H=H, N=N, T=T,
                routing=str(rng.choice(["uniform", "zipf"])), seed=i)


@pytest.mark.parametrize("i", range(N_PRODUCT_CASES))
def test_random_product(i):
    c = draw_product(i)
    try:
        if c["layout"] == "rank":
            import test_gpu_expert_rank as t
            R, T, H, E, K, N = c["R"], c["T"], c["H"], c["E"], c["K"], c["N"]
            if c["fp8"]:
                a, view, d = t.dispatched_fp8(R, T, H, E, K, c["seed"], c["routing"])
                qw, sw = t.fp8_weights(c["seed"] + 1, E, N, H)
            else:
                a, view, d = t.dispatched(R, T, H, E, K, c["seed"], c["routing"])
                wb = t.weights(c["seed"] + 1, E, N, H, 1.0 / np.sqrt(H))
            m = view.plane_stride
            out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            if c["fp8"]:
                a.expert_gemm_rank_fp8(qw, sw, True, out)
            else:
                a.expert_gemm_rank(wb, True, out)
            torch.cuda.synchronize()
            assert a.get_error() == (0, 0)
            got = parity.to_host_u16(out)
            rows = t.valid_rows(d["r"]["recv_counts"], m)
            if c["fp8"]:
                t.check_fp8(got, d, qw, sw, True, rows)
            else:
                t.check(got, d, wb, True, rows)
            counts = d["r"]["recv_counts"]
            for dd in range(R):
                for s in range(R):
                    assert np.isnan(parity.f32(got[dd, s, counts[dd, s]:])).all()
            a.combine(None, False)
        else:
            import test_gpu_expert_gemm as g
            R, T, H, E, K, N = c["R"], c["T"], c["H"], c["E"], c["K"], c["N"]
            if c["fp8"]:
                a, view, d = g.dispatched_fp8(R, T, H, E, K, c["seed"])
                qw, sw = g.fp8_weights(c["seed"] + 1, E, N, H)
            else:
                a, view, d = g.dispatched(R, T, H, E, K, c["seed"], c["routing"])
                wb = g.weights(c["seed"] + 1, E, N, H, 1.0 / np.sqrt(H))
            cap = view.plane_stride
            out = torch.full((E, cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            if c["fp8"]:
                a.expert_gemm_fp8(parity.to_dev(qw, torch.uint8), parity.to_dev(sw, torch.float32),
                                  out)
            else:
                a.expert_gemm(parity.to_dev(wb, torch.bfloat16), out)
            torch.cuda.synchronize()
            assert a.get_error() == (0, 0)
            got = parity.to_host_u16(out)
            counts = d["r"]["recv_counts"]
            if c["fp8"]:
                g.check_rows_fp8(got, d, qw, sw, range(cap))
            else:
                g.check_rows(got, d["rx"], wb, counts, range(cap))
            for e in range(E):
                assert (got[e, counts[e]:] == 0x7FC0).all()
            a.combine(None, False)
    except AssertionError as e:
        raise AssertionError("product case %d %s: %s" % (i, c, e)) from e


# --------------------------------------------------------------------------
# Combine modes on random shapes (rank layout): per-rank token counts with
# dead ranks, the bf16 top-k-slot tree, and the FP8 output (plain and fused).
# --------------------------------------------------------------------------

N_MODE_CASES = 48
MODES = ("varlen-dead", "tree", "out8", "out8-fused")


def draw_mode(i):
    rng = np.random.default_rng(9000 + i)
    mode = MODES[i % len(MODES)]
    R = int(rng.choice([2, 3, 4, 5, 8, 12, 16]))
    Epr = int(rng.integers(1, 9))
    E = R * Epr
    K = int(rng.integers(1, min(8, E) + 1))
    H = int(rng.choice([16, 48, 144, 512, 1040, 2048, 7168]))
    T = int(rng.integers(1, 301))
    while R * R * T * H * 4 > WORKSPACE_BUDGET and T > 1:
        T = max(1, T // 2)
    counts = [int(v) for v in rng.integers(0, T + 1, R)]
    dead = [d for d in range(R) if rng.random() < 0.25][:R - 1]
    return dict(mode=mode, R=R, E=E, K=K, H=H, T=T, counts=counts, dead=dead,
                routing=str(rng.choice(["uniform", "zipf"])),
                weighted=bool(rng.integers(2)) and mode != "tree",
                fused=bool(rng.integers(2)) or mode == "out8-fused", seed=i)


def run_mode(c):
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_REDUCE_BF16_TOPK_TREE
    R, E, K, H, T, seed = c["R"], c["E"], c["K"], c["H"], c["T"], c["seed"]
    ids = synth.topk_ids(seed, R, T, E, K, c["routing"])
    w = synth.topk_weights(seed, R, T, K)
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    res = synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H)
    gam = synth.gamma(seed, H)
    a = MoeA2A(R, T, H, E, K, "cuda")
    dev = parity.to_dev
    live = np.ones((R, T), bool)
    ids_o = ids.copy()
    if c["mode"] == "varlen-dead":
        for s, n in enumerate(c["counts"]):
            ids_o[s, n:] = -1
            live[s, n:] = False
        for d in c["dead"]:
            ids_o[(ids_o >= 0) & (ids_o // (E // R) == d)] = -1
        a.set_active_ranks(((1 << R) - 1) & ~sum(1 << d for d in c["dead"]))
        view = a.dispatch_varlen(dev(ids, torch.int32), dev(w, torch.float32),
                                 dev(x, torch.bfloat16), c["counts"])
    else:
        if c["mode"] == "tree":
            a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
        view = a.dispatch(dev(ids, torch.int32), dev(w, torch.float32), dev(x, torch.bfloat16))
    r = oracle.route(ids_o, w, E, T)
    cnt = view.recv_counts.cpu().numpy()
    assert np.array_equal(cnt, r["recv_counts"]), "recv_counts"
    eo = synth.expert_out_planes(seed, R, T, H, cnt)
    pay = a.combine_payload()
    for d in range(R):
        for s in range(R):
            if cnt[d, s]:
                pay[d, s, :cnt[d, s]].copy_(dev(eo[d, s, :cnt[d, s]], torch.bfloat16))
    fused = c["fused"]
    rout = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    res_d, gam_d = dev(res, torch.bfloat16), dev(gam, torch.bfloat16)
    tok = np.flatnonzero(live.ravel())
    if c["mode"].startswith("out8"):
        if fused:
            out, sc = a.combine_fp8(None, c["weighted"], res_d, gam_d, 1e-6, residual_out=rout)
        else:
            out, sc = a.combine_fp8(None, c["weighted"])
    elif fused:
        out = a.combine(None, c["weighted"], res_d, gam_d, 1e-6, residual_out=rout)
    else:
        out = a.combine(None, c["weighted"])
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 0
    if c["mode"] == "tree":
        oc = oracle.combine_topk_tree(r, ids_o, E, eo, res if fused else None,
                                      gam if fused else None, 1e-6, tokens=tok)
    else:
        oc = oracle.combine(r, eo, c["weighted"], res if fused else None,
                            gam if fused else None, 1e-6, tokens=tok)
    if fused:
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H)[tok],
                              oc["residual_out"]), "residual_out"
    if c["mode"].startswith("out8"):
        g_q = out.view(torch.uint8).cpu().numpy().reshape(R * T, H)[tok]
        g_s = sc.cpu().numpy().ravel()[tok]
        if fused:
            y = oc["y"]
            q_ref, s_ref = oracle.quantize_f32_rows_fp8(y.astype(np.float32))
            assert (np.abs(g_s.astype(np.float64) - s_ref) <= 1e-5 * s_ref).all(), "scales"
            deq = oracle.fp8_to_f32(g_q).astype(np.float64) * g_s[:, None].astype(np.float64)
            bound = (2.0 ** -4 + 1e-4) * np.abs(y) + 2.0 ** -10 * g_s[:, None] + 1e-6
            assert (np.abs(deq - y) <= bound).all(), "FP8 fused output"
        else:
            q_ref, s_ref = oracle.quantize_f32_rows_fp8(oc["acc"])
            assert np.array_equal(g_q, q_ref), "FP8 codes"
            assert np.array_equal(g_s.view(np.uint32), s_ref.view(np.uint32)), "FP8 scales"
    else:
        got = parity.to_host_u16(out).reshape(R * T, H)[tok]
        if fused:
            y = parity.f32(got).astype(np.float64)
            err = np.abs(y - oc["y"])
            assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()
        else:
            assert np.array_equal(got, oc["out"]), "combine sum"
    a.close()


@pytest.mark.parametrize("i", range(N_MODE_CASES))
def test_random_combine_mode(i):
    c = draw_mode(i)
    try:
        run_mode(c)
    except AssertionError as e:
        raise AssertionError("mode case %d %s: %s" % (i, c, e)) from e
