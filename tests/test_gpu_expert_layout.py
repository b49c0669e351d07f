"""Expert-major receive layout (one expert per received row) against the oracle.

InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided NVLink EP for the
GB SKUs": the low-latency padded layouts carry one expert per received row,
and their combine applies the gates in the kernel ("weighted-kernel-sum",
the top-k axis summed in problem order).  Routing tables, counts, source
map, row weights and dispatched rows must equal the oracle bit for bit; the
plain-sum combine and residual_out too; the fused RMSNorm output within the
spec tolerance.
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


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()


def make(R, T, H, E, K, seed, routing="uniform", dup=False):
    ids = synth.topk_ids(seed, R, T, E, K, routing)
    if dup:                                   # repeats and absent ids
        rng = np.random.default_rng(seed)
        ids = rng.integers(-1, E, (R, T, K)).astype(np.int32)
    return dict(ids=ids, w=synth.topk_weights(seed, R, T, K),
                x=synth.per_rank_rows(seed, synth.X, R, T, H),
                res=synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H),
                g=synth.gamma(seed, H))


def run(R, T, H, E, K, seed, weighted, fused, m=None, counts=None, dead=0, dup=False,
        routing="uniform", fp8=False):
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MOE_LAYOUT_EXPERT,
                                                     MOE_FORMAT_FP8_E4M3)
    m = T if m is None else m
    inp = make(R, T, H, E, K, seed, routing, dup)
    a = MoeA2A(R, m, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    a.workspace.fill_(parity.POISON)
    if fp8:
        a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    if dead:
        a.set_active_ranks(((1 << R) - 1) & ~dead)
    dev = parity.to_dev
    ids, w, x = dev(inp["ids"], torch.int32), dev(inp["w"], torch.float32), \
        dev(inp["x"], torch.bfloat16)
    view = a.dispatch_varlen(ids, w, x, counts) if counts is not None else a.dispatch(ids, w, x, m)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    cap = view.plane_stride
    assert cap == R * m and view.layout == MOE_LAYOUT_EXPERT

    # ---- oracle on the ids as the call sees them ----
    ids_o = inp["ids"].copy()
    if counts is not None:
        for s, c in enumerate(counts):
            ids_o[s, c:] = -1
    for d in range(R):
        if dead >> d & 1:
            ids_o[(ids_o >= 0) & (ids_o // (E // R) == d)] = -1
    r = oracle.route_experts(ids_o, inp["w"], E, m)
    cnt = view.recv_counts.cpu().numpy()
    assert np.array_equal(cnt, r["recv_counts"]), "recv_counts"
    assert np.array_equal(view.local_expert_counts.cpu().numpy(), r["local_expert_counts"])
    Tt = view.token_stride
    ss = view.send_slot.cpu().numpy()[:, :T, :K]
    dw = view.dest_weight.cpu().numpy()[:, :T, :K]
    live = np.zeros((R, T), bool)
    for s in range(R):
        live[s, :counts[s] if counts is not None else T] = True
    assert np.array_equal(ss[live], r["send_row"][live]), "send_row"
    assert np.array_equal(dw[live].view(np.uint32), r["wsum"][live].view(np.uint32)), "wsum"
    src = view.src_token.cpu().numpy()
    rw = view.recv_topk_w.cpu().numpy()
    for e in range(E):
        c = cnt[e]
        assert np.array_equal(src[e, :c], r["src_row"][e, :c]), "src_token"
        assert np.array_equal(rw[e, :c].view(np.uint32), r["recv_w"][e, :c].view(np.uint32))
    rows = parity.to_host_u16(view.recv_x) if not fp8 else \
        view.recv_x.view(torch.uint8).cpu().numpy()
    if fp8:
        q_ref, s_ref = oracle.quantize_rows_fp8(inp["x"])
        gs = view.recv_scale.cpu().numpy()
        for e in range(E):
            for j in range(cnt[e]):
                s, t = divmod(int(r["src_row"][e, j]), Tt)
                assert np.array_equal(rows[e, j], q_ref[s, t])
                assert gs[e, j] == s_ref[s, t]
            assert (rows[e, cnt[e]:] == parity.POISON).all()
    else:
        rx = oracle.dispatch_experts(inp["x"], E, m, r,
                                     recv_x=np.full((E, cap, H), 0xFFFF, np.uint16))
        assert np.array_equal(rows, rx), "recv_x (rows and untouched padding)"

    # ---- combine ----
    eo = np.full((E, cap, H), 0x7FC0, np.uint16)
    rng = np.random.default_rng(seed + 1)
    for e in range(E):
        if cnt[e]:
            eo[e, :cnt[e]] = parity.f32_to_bits(
                rng.standard_normal((cnt[e], H)).astype(np.float32))
    pay = a.combine_payload()
    assert tuple(pay.shape) == (E, cap, H)
    pay.copy_(parity.to_dev(eo, torch.bfloat16))
    out = torch.full((R, Tt, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    rout = torch.full_like(out, float("nan")) if fused else None
    res_d = dev(inp["res"], torch.bfloat16) if fused else None
    gam_d = dev(inp["g"], torch.bfloat16) if fused else None
    a.combine(None, weighted, res_d, gam_d, 1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 0
    toks = np.array([s * T + t for s in range(R) for t in range(T) if live[s, t]], np.int64)
    oc = oracle.combine_experts(r, eo, weighted, inp["res"] if fused else None,
                                inp["g"] if fused else None, 1e-6, tokens=toks)
    g = parity.to_host_u16(out).reshape(R * T, H)[toks]
    if not fused:
        assert np.array_equal(g, oc["out"]), "combine (bit-exact)"
    else:
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H)[toks],
                              oc["residual_out"]), "residual_out"
        err = np.abs(parity.f32(g).astype(np.float64) - oc["y"])
        assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"])).all()
    if counts is not None:                     # rows past a count untouched
        o = parity.to_host_u16(out)
        for s, c in enumerate(counts):
            assert (o[s, c:] == 0x7FC0).all()
    return a, view, r


@pytest.mark.parametrize("weighted,fused", [(False, False), (True, False), (False, True),
                                            (True, True)])
def test_expert_layout_variants_ragged(weighted, fused):
    # H = 136 (not a multiple of 64), K = 5, repeats and -1 ids
    run(6, 100, 136, 48, 5, 3, weighted, fused, dup=True)


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
def test_expert_layout_top_k_instantiations(K):
    # top-k values with their own routing instantiation (1, 2, 4, 8) and a
    # generic one (3); repeats and -1 ids; three tiles on one source
    run(3, 530, 64, 24, K, 50 + K, True, True, dup=True)


def test_expert_layout_decode_shape():
    a, view, r = run(8, 64, 7168, 256, 8, 0, True, True)
    # every token has 8 distinct experts: 8 rows per token
    assert view.recv_counts.sum().item() == 8 * 64 * 8


def test_expert_layout_many_tiles_and_sources():
    # three 256-token tiles per source: the row bases run across tiles and sources
    run(4, 600, 64, 64, 8, 5, True, False, routing="zipf")


def test_expert_layout_runtime_max_above_tokens():
    run(4, 40, 128, 32, 4, 6, True, True, m=56)


def test_expert_layout_limits():
    # the layout's largest expert count (1024, lane masks in shared memory),
    # 32 ranks and top-32 (32 send-table entries per token), long rows
    run(8, 70, 64, 1024, 8, 41, True, True)
    run(32, 12, 64, 64, 32, 42, True, True)
    run(2, 10, 16384, 4, 2, 43, True, True)


def test_expert_layout_single_rank():
    run(1, 300, 128, 8, 2, 44, True, True)


def test_expert_layout_varlen_and_dead_rank():
    run(8, 96, 256, 64, 8, 7, True, True, counts=[96, 0, 5, 95, 1, 64, 33, 96], dead=0b100100)


def test_expert_layout_fp8_rows():
    run(4, 80, 256, 32, 8, 8, True, False, fp8=True)


def test_expert_layout_rejects_tree_and_large_E():
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MoeA2AError, MOE_LAYOUT_EXPERT,
                                                     MOE_REDUCE_BF16_TOPK_TREE)
    a = MoeA2A(2, 8, 64, 4, 2, "cuda", layout=MOE_LAYOUT_EXPERT)
    with pytest.raises(MoeA2AError):
        a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
    with pytest.raises(MoeA2AError):
        MoeA2A(2, 8, 64, 2048, 2, "cuda", layout=MOE_LAYOUT_EXPERT)


@pytest.mark.parametrize("fused", [False, True])
def test_expert_layout_fp8_combine_output(fused):
    # the FP8 combine output in the expert layout: plain sum bit for bit,
    # fused RMSNorm output within one e4m3 step of the oracle's quantisation
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_LAYOUT_EXPERT
    R, T, H, E, K = 4, 90, 256, 32, 6
    inp = make(R, T, H, E, K, 21, dup=True)
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    dev = parity.to_dev
    view = a.dispatch(dev(inp["ids"], torch.int32), dev(inp["w"], torch.float32),
                      dev(inp["x"], torch.bfloat16))
    r = oracle.route_experts(inp["ids"], inp["w"], E, T)
    cnt = view.recv_counts.cpu().numpy()
    cap = view.plane_stride
    eo = np.full((E, cap, H), 0x7FC0, np.uint16)
    rng = np.random.default_rng(22)
    for e in range(E):
        if cnt[e]:
            eo[e, :cnt[e]] = parity.f32_to_bits(rng.standard_normal((cnt[e], H)).astype(np.float32))
    a.combine_payload().copy_(dev(eo, torch.bfloat16))
    res = dev(inp["res"], torch.bfloat16) if fused else None
    gam = dev(inp["g"], torch.bfloat16) if fused else None
    out, sc = a.combine_fp8(None, True, res, gam, 1e-6)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    oc = oracle.combine_experts(r, eo, True, inp["res"] if fused else None,
                                inp["g"] if fused else None, 1e-6)
    g_q = out.view(torch.uint8).cpu().numpy().reshape(R * T, H)
    g_s = sc.cpu().numpy().ravel()
    if not fused:
        q_ref, s_ref = oracle.quantize_f32_rows_fp8(oc["acc"])
        assert np.array_equal(g_q, q_ref)
        assert np.array_equal(g_s.view(np.uint32), s_ref.view(np.uint32))
    else:
        q_ref, s_ref = oracle.quantize_f32_rows_fp8(oc["y"].astype(np.float32))
        assert (np.abs(g_s.astype(np.float64) - s_ref) <= 1e-5 * s_ref).all()
        step = lambda c: np.where(c & 0x80, -(c.astype(np.int32) & 0x7F), c.astype(np.int32) & 0x7F)
        assert (np.abs(step(g_q) - step(q_ref)) <= 1).all()


@pytest.mark.parametrize("small_max", ["-1", "256"])
@pytest.mark.parametrize("T", [1, 33, 64, 200, 256])
def test_expert_one_launch_dispatch_modes(monkeypatch, small_max, T):
    # the same batches through the routing passes + row copy (-1) and the
    # one-launch dispatch (up to 256 tokens per rank): both equal the oracle
    # (routing tables, counts, rows, untouched padding, combines)
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_LAYOUT_EXPERT
    monkeypatch.setenv("MOE_DISPATCH_SMALL_MAX", small_max)
    run(8, T, 256, 64, 8, seed=T + 7, weighted=True, fused=True)
    run(4, T, 128, 16, 4, seed=T + 8, weighted=False, fused=False, routing="zipf")
    a = MoeA2A(4, T, 128, 16, 4, "cuda", layout=MOE_LAYOUT_EXPERT)
    view = a.dispatch(parity.to_dev(synth.topk_ids(1, 4, T, 16, 4), torch.int32),
                      parity.to_dev(synth.topk_weights(1, 4, T, 4), torch.float32),
                      torch.zeros((4, T, 128), dtype=torch.bfloat16, device="cuda"))
    assert view.kernels == (3 if small_max == "-1" else 1)
    a.combine(None, False)


def test_expert_one_launch_alternates_with_the_routing_passes():
    # One handle, calls alternating between the one-launch dispatch (T <= 256)
    # and the routing passes (T = 300), with ranks marked dead and alive again
    # in between: every call's rows per expert and histogram are the
    # oracle's (the one-launch path adds into a buffer pair that the previous
    # call cleared; the routing passes write the first pair).
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_LAYOUT_EXPERT
    R, M, H, E, K = 4, 300, 128, 16, 4
    a = MoeA2A(R, M, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    plan = [(40, 0), (40, 0), (300, 0), (17, 0b0100), (300, 0b0010), (64, 0), (1, 0), (40, 0)]
    for n, (T, dead) in enumerate(plan):
        a.set_active_ranks(((1 << R) - 1) & ~dead)
        inp = make(R, T, H, E, K, seed=100 + n)
        view = a.dispatch(parity.to_dev(inp["ids"], torch.int32),
                          parity.to_dev(inp["w"], torch.float32),
                          parity.to_dev(inp["x"], torch.bfloat16))
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0)
        assert view.kernels == (1 if T <= 256 else 3), (n, T)
        ids_o = inp["ids"].copy()
        for d in range(R):
            if dead >> d & 1:
                ids_o[(ids_o >= 0) & (ids_o // (E // R) == d)] = -1
        r = oracle.route_experts(ids_o, inp["w"], E, T)
        assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"]), (n, T)
        assert np.array_equal(view.local_expert_counts.cpu().numpy(),
                              r["local_expert_counts"]), (n, T)
        ss = view.send_slot.cpu().numpy()[:, :T, :K]
        assert np.array_equal(ss, r["send_row"]), (n, T)
        a.combine(None, False)


@pytest.mark.parametrize("small_max", ["-1", "256"])
@pytest.mark.parametrize("T", [1, 40, 128, 200])
def test_expert_fp8_one_launch_dispatch_modes(monkeypatch, small_max, T):
    # FP8 receive rows on the expert layout, through the routing passes + FP8
    # row copy (-1) and the one-launch dispatch (one CTA per token): codes,
    # scales, routing tables and combines equal the oracle on both
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MOE_LAYOUT_EXPERT,
                                                     MOE_FORMAT_FP8_E4M3)
    monkeypatch.setenv("MOE_DISPATCH_SMALL_FP8_MAX", small_max)
    run(8, T, 256, 64, 8, seed=T + 9, weighted=True, fused=True, fp8=True)
    run(4, T, 7168, 16, 3, seed=T + 10, weighted=False, fused=False, fp8=True, routing="zipf")
    a = MoeA2A(4, T, 128, 16, 4, "cuda", layout=MOE_LAYOUT_EXPERT)
    a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    view = a.dispatch(parity.to_dev(synth.topk_ids(2, 4, T, 16, 4), torch.int32),
                      parity.to_dev(synth.topk_weights(2, 4, T, 4), torch.float32),
                      torch.zeros((4, T, 128), dtype=torch.bfloat16, device="cuda"))
    assert view.kernels == (3 if small_max == "-1" else 1)
    a.combine(None, False)
