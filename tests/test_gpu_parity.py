"""CUDA path vs oracle, through the C ABI, on the five workloads.

Small cases are compared in full; the full-size workloads (decode, prefill,
wide EP, every ladder rung) run in the same launch configuration as the
benchmark and are compared in full for routing, counts, slot maps, metadata
and dispatched rows, and on a seeded sample of tokens (plus edge tokens) for
the combine, which the oracle computes token by token.
"""
import numpy as np
import pytest

from combine_topk_ids_rank_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()


def small(name, **kw):
    from dataclasses import replace
    return replace(synth.WORKLOADS[name], **kw)


def test_tiny():
    rep = parity.Case(synth.WORKLOADS["tiny"]).run()
    assert rep["tokens_checked"] == 32


@pytest.mark.parametrize("weighted,fused", [(False, False), (True, False), (False, True),
                                            (True, True)])
def test_variants_small(weighted, fused):
    # ragged: T not a multiple of the 256-token routing tile, H=136 not a
    # multiple of the 64-element vector span of a warp, R not a multiple of 4
    w = small("decode", ep_size=6, tokens_per_rank=300, max_tokens=320, runtime_max=310,
              hidden=136, num_experts=48, top_k=5, weighted=weighted, fused=fused)
    parity.Case(w).run(seed=3)


@pytest.mark.parametrize("overlap", ["0", "1"])
def test_route_overlap_modes(monkeypatch, overlap):
    # Three 256-token routing tiles per source plus a ragged tail.  "1" (the
    # default): the row copy starts after the first routing pass and adds
    # each tile's prefix to the token's tile-local slots while the second
    # pass runs on the handle's own stream; "0": the passes run in stream
    # order in front of the copy.  Both must equal the oracle.
    monkeypatch.setenv("MOE_ROUTE_OVERLAP", overlap)
    w = small("decode", ep_size=6, tokens_per_rank=700, max_tokens=720, runtime_max=710,
              hidden=136, num_experts=48, top_k=5, weighted=True, fused=True)
    parity.Case(w).run(seed=11)


@pytest.mark.parametrize("small_max", ["-1", "0"])
@pytest.mark.parametrize("T", [1, 33, 64, 256])
def test_one_launch_dispatch_modes(monkeypatch, small_max, T):
    # Batches of at most one 256-token routing tile per source: "0" (the
    # default, up to 256 tokens) dispatches in one launch, each copy warp deriving its token's
    # slots from the ids before it; "-1" forces the two routing passes and the
    # row copy.  Both must equal the oracle (rows chunked when tokens are few).
    monkeypatch.setenv("MOE_DISPATCH_SMALL_MAX", small_max)
    w = small("decode", ep_size=6, tokens_per_rank=T, max_tokens=260, runtime_max=T + 3,
              hidden=1032, num_experts=48, top_k=5, weighted=True, fused=True)
    rep = parity.Case(w).run(seed=T)
    assert rep["kernels"] == (1 if small_max == "0" and T <= 256 else 3)


@pytest.mark.parametrize("small_max", ["-1", "4096"])
@pytest.mark.parametrize("R,T,H,E,K,weighted,fused", [
    (6, 33, 136, 48, 5, True, True), (6, 33, 136, 48, 5, False, False),
    (8, 64, 7168, 256, 8, True, True), (4, 20, 16384, 16, 4, True, True),
    (32, 8, 64, 256, 32, False, True), (8, 128, 1032, 64, 8, True, False)])
def test_cluster_combine_modes(monkeypatch, small_max, R, T, H, E, K, weighted, fused):
    # "4096" combines each token of these calls on a cluster of CTAs, each
    # owning a column slice, the fused sum of squares exchanged through
    # distributed shared memory (the default does so up to 64 tokens); "-1"
    # forces the persistent combines.  Both must equal the oracle (ragged
    # slices at H = 136, two vectors per thread at H = 16384, 32 ranks).
    monkeypatch.setenv("MOE_COMBINE_SMALL_MAX", small_max)
    w = small("decode", ep_size=R, tokens_per_rank=T, max_tokens=T, runtime_max=T, hidden=H,
              num_experts=E, top_k=K, weighted=weighted, fused=fused)
    parity.Case(w).run(seed=T + H)


def test_one_launch_and_two_pass_dispatches_interleaved():
    # One handle, batches alternating between the one-launch dispatch (which
    # alternates two local-expert count buffers between calls) and the
    # two-pass routing (T > 256): every call's counts and tables must be the
    # oracle's.
    w = small("decode", ep_size=4, tokens_per_rank=600, max_tokens=600, runtime_max=600,
              hidden=256, num_experts=32, top_k=4, weighted=True, fused=True)
    case = parity.Case(w)
    for T in (64, 40, 600, 7, 64, 300, 33, 33):
        case.run(T=T, seed=T)


@pytest.mark.parametrize("K", [1, 2, 4, 8, 3])
def test_top_k_variants(K):
    w = small("decode", ep_size=4, tokens_per_rank=77, max_tokens=80, runtime_max=80,
              hidden=64, num_experts=32, top_k=K)
    parity.Case(w).run(seed=K)


# The handle's limits (MOE_MAX_EP_SIZE 32, MOE_MAX_TOP_K 32, MOE_MAX_HIDDEN
# 16384, MOE_MAX_EXPERTS 8192) and the row lengths where the combine's
# vectors per thread change (4096 -> 4104, 7168 -> 7176).
@pytest.mark.parametrize("fused", [False, True])
def test_limit_32_ranks_top_32(fused):
    w = small("decode", ep_size=32, tokens_per_rank=40, max_tokens=48, runtime_max=44,
              hidden=64, num_experts=256, top_k=32, weighted=True, fused=fused)
    parity.Case(w).run(seed=5)


@pytest.mark.parametrize("weighted,fused", [(False, False), (True, True)])
def test_limit_hidden_16384(weighted, fused):
    w = small("decode", ep_size=2, tokens_per_rank=20, max_tokens=24, runtime_max=20,
              hidden=16384, num_experts=4, top_k=2, weighted=weighted, fused=fused)
    parity.Case(w).run(seed=6)


@pytest.mark.parametrize("weighted,fused", [(False, False), (True, True)])
def test_single_rank(weighted, fused):
    # ep_size 1: every expert is local, one plane, three routing tiles
    w = small("decode", ep_size=1, tokens_per_rank=600, max_tokens=600, runtime_max=600,
              hidden=256, num_experts=16, top_k=4, weighted=weighted, fused=fused)
    parity.Case(w).run(seed=9)


def test_limit_8192_experts():
    w = small("decode", ep_size=8, tokens_per_rank=300, max_tokens=300, runtime_max=300,
              hidden=64, num_experts=8192, top_k=8)
    parity.Case(w).run(seed=7)


@pytest.mark.parametrize("H", [4096, 4104, 7168, 7176, 8192])
def test_hidden_at_vector_boundaries(H):
    w = small("decode", ep_size=4, tokens_per_rank=33, max_tokens=40, runtime_max=36,
              hidden=H, num_experts=16, top_k=4)
    parity.Case(w).run(seed=H % 97)


def test_decode():
    rep = parity.Case(synth.WORKLOADS["decode"]).run()
    assert rep["tokens_checked"] == 512


def test_prefill_zipf():
    # every token of the full-size batch, element by element
    rep = parity.Case(synth.WORKLOADS["prefill"]).run(sample=None)
    assert rep["tokens_checked"] == 8 * 4096 and rep["padding_checked"]
    # Zipf(1.2) with contiguous placement: ~2.9 destination ranks per token
    assert 2.7 < rep["recv_rows"] / (8 * 4096) < 3.1


def test_wide_ep():
    rep = parity.Case(synth.WORKLOADS["wide"]).run(sample=None)
    assert rep["tokens_checked"] == 16 * 1024 and rep["padding_checked"]
    assert 6.3 < rep["recv_rows"] / (16 * 1024) < 6.7


def test_ladder_all_rungs_one_workspace():
    w = synth.WORKLOADS["ladder"]
    case = parity.Case(w)                       # sized once for 8192 tokens/rank
    inputs = synth.inputs(w, seed=0)            # rung T uses the first T tokens
    from oracle import oracle
    r_big = oracle.route(inputs["topk_ids"], inputs["topk_w"], w.num_experts, w.max_tokens)
    big_eo = synth.expert_out_planes(0, w.ep_size, w.max_tokens, w.hidden,
                                     r_big["recv_counts"])
    for T in synth.LADDER_RUNGS:
        # every token of every rung, element by element
        rep = case.run(T=T, inputs=inputs, big_eo=big_eo, sample=None)
        assert rep["T"] == T and rep["tokens_checked"] == 8 * T


def test_repeat_calls_bit_identical():
    w = small("decode", tokens_per_rank=40, max_tokens=64, runtime_max=48, hidden=256)
    case = parity.Case(w)
    inp = synth.inputs(w, 5)
    outs = []
    for _ in range(3):
        view = case.a2a.dispatch(parity.to_dev(inp["topk_ids"], torch.int32),
                                 parity.to_dev(inp["topk_w"], torch.float32),
                                 parity.to_dev(inp["x"], torch.bfloat16), w.runtime_max)
        res = parity.to_dev(inp["residual"], torch.bfloat16)
        out = case.a2a.combine(view.recv_x, True, res,
                               parity.to_dev(inp["gamma"], torch.bfloat16), 1e-6)
        outs.append(parity.to_host_u16(out))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# --------------------------------------------------------------------------
# Compatibility reduction (bf16 tree over top-k slots) against its oracle
# --------------------------------------------------------------------------

def _tree_case(R, T, H, E, K, seed, fused, ids=None, eo_fn=None):
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_REDUCE_BF16_TOPK_TREE
    from oracle import oracle
    ids = synth.topk_ids(seed, R, T, E, K) if ids is None else ids
    w = synth.topk_weights(seed, R, T, K)
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    a = MoeA2A(R, T, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)
    a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
    view = a.dispatch(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                      parity.to_dev(x, torch.bfloat16))
    counts = view.recv_counts.cpu().numpy()
    r = oracle.route(ids, w, E, T)
    if eo_fn is None:
        eo = synth.expert_out_planes(seed, R, T, H, counts)
    else:
        eo = np.full((R, R, T, H), 0x7FC0, np.uint16)
        for d in range(R):
            for s in range(R):
                eo[d, s, :counts[d, s]] = parity.f32_to_bits(eo_fn(d))
    pay = a.combine_payload()
    for d in range(R):
        for s in range(R):
            c = int(counts[d, s])
            if c:
                pay[d, s, :c].copy_(parity.to_dev(eo[d, s, :c], torch.bfloat16))
    res = synth.per_rank_rows(seed, synth.RESIDUAL, R, T, H) if fused else None
    gam = synth.gamma(seed, H) if fused else None
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out) if fused else None
    a.combine(None, False, parity.to_dev(res, torch.bfloat16) if fused else None,
              parity.to_dev(gam, torch.bfloat16) if fused else None, 1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    oc = oracle.combine_topk_tree(r, ids, E, eo, res, gam, 1e-6)
    g = parity.to_host_u16(out).reshape(R * T, H)
    if not fused:
        assert np.array_equal(g, oc["out"])
    else:
        assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"])
        err = np.abs(parity.f32(g).astype(np.float64) - oc["y"])
        assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"])).all()
    return parity.f32(g)


def test_topk_tree_pages_probe_on_gpu():
    # {1.0, 7 x 2^-9} over eight slots -> 1.0078125 (the bf16 tree's value)
    R = 8
    ids = np.tile(np.arange(R, dtype=np.int32), (R, 1, 1)).reshape(R, 1, R)
    vals = [1.0] + [2.0 ** -9] * 7
    out = _tree_case(R, 1, 64, R, R, 0, False, ids=ids,
                     eo_fn=lambda d: np.full(64, vals[d], np.float32))
    assert np.all(out == 1.0078125)


@pytest.mark.parametrize("fused", [False, True])
def test_topk_tree_decode_shape(fused):
    _tree_case(8, 64, 7168, 256, 8, 3, fused)


def test_topk_tree_duplicates_and_missing_ids():
    R, T, E, K = 4, 70, 16, 6
    rng = np.random.default_rng(4)
    ids = rng.integers(-1, E, (R, T, K)).astype(np.int32)   # repeats and -1
    _tree_case(R, T, 200, E, K, 4, True, ids=ids)


def test_topk_tree_rejects_weighted():
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MoeA2AError,
                                                     MOE_REDUCE_BF16_TOPK_TREE,
                                                     MOE_ERR_INVALID_ARG)
    a = MoeA2A(2, 8, 64, 4, 2, "cuda")
    a.set_reduction(MOE_REDUCE_BF16_TOPK_TREE)
    ids = parity.to_dev(synth.topk_ids(0, 2, 8, 4, 2), torch.int32)
    w = parity.to_dev(synth.topk_weights(0, 2, 8, 2), torch.float32)
    v = a.dispatch(ids, w, torch.zeros((2, 8, 64), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(MoeA2AError) as e:
        a.combine(v.recv_x, True)
    assert e.value.status == MOE_ERR_INVALID_ARG and a.phase == 1
    a.combine(v.recv_x, False)
