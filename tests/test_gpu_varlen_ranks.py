"""Per-rank token counts and dead ranks, against the oracle.

Readings (the pages name these features, not their arithmetic): a token
past its rank's count is absent, exactly as if all its expert ids were -1;
an expert that lives on a dead rank is treated as an absent expert; a rank
marked dead after dispatch is skipped by combine.  So the oracle runs on the
masked ids (or, for a rank lost between the phases, on the routing with that
rank removed) and the CUDA path must match it bit for bit / within the
RMSNorm tolerance.
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

R, M, H, E, K = 8, 96, 384, 64, 8


def inputs(seed, m=M):
    return dict(ids=synth.topk_ids(seed, R, m, E, K), w=synth.topk_weights(seed, R, m, K),
                x=synth.per_rank_rows(seed, synth.X, R, m, H),
                res=synth.per_rank_rows(seed, synth.RESIDUAL, R, m, H), g=synth.gamma(seed, H))


def masked(ids, counts=None, dead=()):
    ids = ids.copy()
    if counts is not None:
        for s, c in enumerate(counts):
            ids[s, c:] = -1
    for d in dead:
        ids[(ids >= 0) & (ids // (E // R) == d)] = -1
    return ids


def run_gpu(a, inp, counts=None, weighted=True, after_dispatch=None):
    dev = lambda v, dt: parity.to_dev(v, dt)
    ids, w, x = dev(inp["ids"], torch.int32), dev(inp["w"], torch.float32), dev(inp["x"], torch.bfloat16)
    view = a.dispatch_varlen(ids, w, x, counts) if counts is not None else a.dispatch(ids, w, x)
    m = view.plane_stride
    cnt = view.recv_counts.cpu().numpy()
    eo = synth.expert_out_planes(7, R, m, H, cnt)
    pay = a.combine_payload()
    for d in range(R):
        for s in range(R):
            if cnt[d, s]:
                pay[d, s, :cnt[d, s]].copy_(dev(eo[d, s, :cnt[d, s]], torch.bfloat16))
    if after_dispatch is not None:
        after_dispatch()
    out = torch.full((R, M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    rout = torch.full_like(out, float("nan"))
    a.combine(None, weighted, dev(inp["res"], torch.bfloat16), dev(inp["g"], torch.bfloat16),
              1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    return view, eo, parity.to_host_u16(out), parity.to_host_u16(rout)


def check(view, eo, out, rout, inp, ids_oracle, tokens, weighted=True, drop_ranks=()):
    r = oracle.route(ids_oracle, inp["w"], E, M)
    # The dispatch ran with every rank of ids_oracle alive: its tables and
    # counts are the full routing's, also when a rank is lost afterwards.
    send_at_dispatch = r["send_slot"].copy()
    cnt = view.recv_counts.cpu().numpy()
    assert np.array_equal(cnt, r["recv_counts"])
    assert np.array_equal(view.local_expert_counts.cpu().numpy(), r["local_expert_counts"])
    for d in drop_ranks:                       # a rank lost between the phases:
        r["dmask"] &= ~np.uint32(1 << d)       # the combine skips its messages
        r["send_slot"][:, :, d] = -1
    ss = view.send_slot.cpu().numpy()[:, :, :R]
    od = oracle.dispatch(ids_oracle, inp["w"], inp["x"], E, M, r)
    rx = parity.to_host_u16(view.recv_x)
    for d in range(R):
        for s in range(R):
            c = cnt[d, s]
            assert np.array_equal(rx[d, s, :c], od["recv_x"][d, s, :c])
            assert np.array_equal(view.recv_topk_ids.cpu().numpy()[d, s, :c], od["recv_ids"][d, s, :c])
    oc = oracle.combine(r, eo, weighted, inp["res"], inp["g"], 1e-6)
    flat = [s * M + t for s, t in tokens]
    assert np.array_equal(rout.reshape(R * M, H)[flat], oc["residual_out"][flat])
    y = parity.f32(out.reshape(R * M, H)[flat]).astype(np.float64)
    err = np.abs(y - oc["y"][flat])
    assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"][flat])).all()
    for s, t in tokens:
        assert np.array_equal(ss[s, t], send_at_dispatch[s, t])


def test_varlen_counts_match_masked_uniform_routing():
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    inp = inputs(1)
    counts = [0, 1, 95, 96, 40, 64, 33, 17]
    a = MoeA2A(R, M, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)
    view, eo, out, rout = run_gpu(a, inp, counts)
    tokens = [(s, t) for s in range(R) for t in range(counts[s])]
    check(view, eo, out, rout, inp, masked(inp["ids"], counts), tokens)
    # rows past each count are left untouched
    for s in range(R):
        assert np.isnan(parity.f32(out[s, counts[s]:])).all()
        assert np.isnan(parity.f32(rout[s, counts[s]:])).all()


def test_dead_ranks_receive_nothing():
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    inp = inputs(2)
    a = MoeA2A(R, M, H, E, K, "cuda")
    a.set_active_ranks(0xFF & ~((1 << 2) | (1 << 5)))
    view, eo, out, rout = run_gpu(a, inp)
    cnt = view.recv_counts.cpu().numpy()
    assert cnt[2].sum() == 0 and cnt[5].sum() == 0
    tokens = [(s, t) for s in range(R) for t in range(M)]
    check(view, eo, out, rout, inp, masked(inp["ids"], dead=(2, 5)), tokens)


def test_rank_lost_between_dispatch_and_combine():
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    inp = inputs(3)
    a = MoeA2A(R, M, H, E, K, "cuda")
    view, eo, out, rout = run_gpu(a, inp, after_dispatch=lambda: a.set_active_ranks(0xFF & ~(1 << 3)))
    tokens = [(s, t) for s in range(R) for t in range(M)]
    check(view, eo, out, rout, inp, inp["ids"], tokens, drop_ranks=(3,))


def test_varlen_with_dead_rank_and_tree_reduction():
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_REDUCE_BF16_TOPK_TREE
    inp = inputs(4)
    counts = [96, 0, 50, 7, 96, 80, 1, 30]
    a = MoeA2A(R, M, H, E, K, "cuda")
    a.set_active_ranks(0xFF & ~(1 << 6))
    a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
    view, eo, out, rout = run_gpu(a, inp, counts, weighted=False)
    ids_o = masked(inp["ids"], counts, dead=(6,))
    r = oracle.route(ids_o, inp["w"], E, M)
    oc = oracle.combine_topk_tree(r, ids_o, E, eo, inp["res"], inp["g"], 1e-6)
    flat = [s * M + t for s in range(R) for t in range(counts[s])]
    assert np.array_equal(rout.reshape(R * M, H)[flat], oc["residual_out"][flat])
