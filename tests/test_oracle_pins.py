"""Pins of the CPU oracle to facts outside itself.

Each test fixes the oracle against a value the pages print (tests/golden/),
a closed form, a brute-force enumeration of the definition, an invariant, or
a library routine in a special case where the method reduces to it.  None of
them re-types the oracle's own loops.  tests/test_oracle_mutants.py plants
mistakes in copies of the oracle and checks that these pins catch them.
"""
import math

import numpy as np
import pytest

from conftest import read_golden, read_golden_table

F32 = np.float32


def bits(values):
    import torch
    t = torch.tensor(np.asarray(values, dtype=np.float32).ravel())
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(np.shape(values))


def f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def route_to_ranks(dest_lists, R, E, K):
    """topk ids for tokens of source 0..: dest_lists[s][t] = list of ranks, one
    expert per listed rank (the first expert of that rank), padded with -1."""
    Epr = E // R
    T = max(len(x) for x in dest_lists)
    ids = np.full((R, T, K), -1, np.int32)
    for s, toks in enumerate(dest_lists):
        for t, ranks in enumerate(toks):
            for k, d in enumerate(ranks):
                ids[s, t, k] = d * Epr
    return ids


def planes_with(routing, R, m, H, value_fn):
    """expert_out [R,R,m,H] whose valid slot (d,s,j) holds value_fn(d,s,j)."""
    eo = np.full((R, R, m, H), 0x7FC0, np.uint16)    # NaN in padding
    for d in range(R):
        for s in range(R):
            for j in range(routing["recv_counts"][d, s]):
                eo[d, s, j, :] = bits(np.full(H, value_fn(d, s, j), np.float32))
    return eo


# --------------------------------------------------------------------------
# bf16 narrowing: a library routine (torch's round-to-nearest-even) pins it
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_library_routine(oracle):
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    vals = vals[~np.isnan(vals)]
    # exact ties, subnormals, overflow edge, infinities, signed zeros
    extra = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130,
                      3.3895314e38, 3.4e38, np.inf, -np.inf, 0.0, -0.0,
                      1.013671875, 255.0], np.float32)
    vals = np.concatenate([vals, extra])
    got = oracle.bf16_bits(vals)
    assert np.array_equal(got, bits(vals))
    nan = oracle.bf16_bits(np.array([np.nan], np.float32))
    assert np.isnan(f32(nan)).all()


def test_bf16_widening_is_exact(oracle):
    allb = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    finite = ~np.isnan(f32(allb))
    import torch
    ref = torch.from_numpy(allb.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    h = oracle.lib()
    got = np.array([h.oracle_f32_from_bf16(int(b)) for b in allb[finite][::7]], np.float32)
    assert np.array_equal(got, ref[finite][::7])


# --------------------------------------------------------------------------
# The pages' probes (tests/golden)
# --------------------------------------------------------------------------

def test_probe_pow2_rank_sum_is_255(oracle):
    g = read_golden("pow2_rank_sum.txt")
    R = int(g["ep_size"])
    E, K, H, T = R, R, 136, 1          # one expert per rank, TOPK = world
    ids = route_to_ranks([[list(range(R))] * T for _ in range(R)], R, E, K)
    w = np.full(ids.shape, 1.0 / K, np.float32)
    r = oracle.route(ids, w, E, T)
    eo = planes_with(r, R, T, H, lambda d, s, j: 2.0 ** d)
    c = oracle.combine(r, eo, weighted=False)
    assert np.all(f32(c["out"]) == float(g["combined"]))
    assert np.all(c["acc"] == F32(float(g["combined"])))


def _tree_bf16(vals, narrow):
    """The pages' hand-unrolled pairwise tree over eight top-k slots with a
    bf16 rounding after every add (((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)))."""
    a = list(vals)
    for stride in (1, 2, 4):
        for i in range(0, 8, 2 * stride):
            a[i] = narrow(a[i] + a[i + stride])
    return a[0]


def test_probe_reduction_discriminator(oracle):
    g = read_golden("reduction_discriminator.txt")
    contribs = [float(eval(v, {})) for v in g["contributions"].split(",")]
    R = len(contribs)
    E, K, H = R, R, 8
    ids = route_to_ranks([[list(range(R))] for _ in range(R)], R, E, K)
    r = oracle.route(ids, np.full(ids.shape, 0.125, np.float32), E, 1)
    eo = planes_with(r, R, 1, H, lambda d, s, j: contribs[d])
    c = oracle.combine(r, eo, weighted=False)
    adopted = float(g[g["adopted"]])
    assert np.all(f32(c["out"]) == adopted)                       # 1.015625
    # The probe discriminates: the other two models give the other printed values.
    narrow = lambda v: float(f32(oracle.bf16_bits(np.array([v], np.float32)))[0])
    assert _tree_bf16(contribs, narrow) == float(g["bf16_tree"])
    seq = 0.0
    for v in contribs:
        seq = narrow(seq + v)
    assert seq == float(g["sequential_bf16"])
    assert len({adopted, float(g["bf16_tree"]), float(g["sequential_bf16"])}) == 3


def test_probe_slot_order_is_ascending_token(oracle):
    g = read_golden("slot_order_probe.txt")
    T, R = int(g["tokens"]), int(g["ep_size"])
    E, K, H = R, R, 16
    ids = route_to_ranks([[list(range(R))] * T for _ in range(R)], R, E, K)
    r = oracle.route(ids, np.full(ids.shape, 0.125, np.float32), E, T)
    eo = planes_with(r, R, T, H, lambda d, s, j: float(j))
    c = oracle.combine(r, eo, weighted=False)
    expect = [float(v) for v in g["expect"].split(",")]
    got_fi = [float(v) for v in g["got_flashinfer"].split(",")]
    for s in range(R):
        per_token = f32(c["out"][s * T:(s + 1) * T, 0])
        assert list(per_token) == expect
        assert np.all(f32(c["out"][s * T:(s + 1) * T]) == per_token[:, None])
    # the total is conserved under any per-rank permutation, so it cannot tell
    assert sum(expect) == sum(got_fi) == float(g["total"])


def test_probe_partial_routing_and_duplicates(oracle):
    g = read_golden("routing_probes.txt")
    R, E, K, H = 4, 16, 3, 24
    Epr = E // R
    # tokens alternate between destination pairs {0,2} and {1,3}; token 2 puts
    # all three experts on rank 3 (duplicates on one rank).
    ids = np.full((R, 6, K), -1, np.int32)
    for s in range(R):
        for t in range(6):
            if t == 2:
                ids[s, t] = [3 * Epr, 3 * Epr + 1, 3 * Epr + 1]
            elif t % 2 == 0:
                ids[s, t, :2] = [0 * Epr + t % Epr, 2 * Epr + 1]
            else:
                ids[s, t, :2] = [1 * Epr, 3 * Epr + 2]
    r = oracle.route(ids, np.full(ids.shape, 0.5, np.float32), E, 6)
    # compaction: each plane holds only the tokens routed there, in order
    assert list(r["src_token"][0, 0, :3]) == [0, 4, -1]
    assert list(r["src_token"][3, 0, :4]) == [1, 2, 3, 5]
    x = np.full((R, 6, H), bits(np.float32(1.0)), np.uint16)
    d = oracle.dispatch(ids, np.full(ids.shape, 0.5, np.float32), x, E, 6, r)
    c = oracle.combine(r, d["recv_x"], weighted=False)
    out = f32(c["out"]).reshape(R, 6, H)
    two = float(g["partial_routing_two_destinations"])
    one = float(g["duplicate_experts_one_rank"])
    for t in range(6):
        assert np.all(out[:, t] == (one if t == 2 else two))


# --------------------------------------------------------------------------
# Statistics of routing against a closed form and the pages' counts
# --------------------------------------------------------------------------

def expected_distinct(R, E, K):
    """Expected number of distinct owner ranks of K distinct uniform experts:
    a rank is missed iff all K experts avoid its E/R experts."""
    return R * (1.0 - math.comb(E - E // R, K) / math.comb(E, K))


@pytest.mark.parametrize("R,E,K,T,expected", [(8, 256, 8, 8192, 5.2947),
                                              (16, 512, 8, 1024, 6.4876),
                                              (2, 8, 2, 16, 1.5714)])
def test_mean_distinct_ranks_closed_form(oracle, R, E, K, T, expected):
    from combine_topk_ids_rank_gb300 import synth
    assert abs(expected_distinct(R, E, K) - expected) < 1e-4
    ids = synth.topk_ids(0, R, T, E, K, "uniform")
    r = oracle.route(ids, synth.topk_weights(0, R, T, K), E, T)
    n = R * T
    per_token = np.array([bin(int(v)).count("1") for v in r["dmask"].ravel()])
    assert r["recv_counts"].sum() == per_token.sum()
    se = per_token.std() / math.sqrt(n)
    assert abs(per_token.mean() - expected) < max(5 * se, 1e-9)


def test_pages_recv_counts_match_closed_form():
    rows = read_golden_table("recv_counts_ep8_top8.txt")
    mu = expected_distinct(8, 256, 8)
    # the standard deviation of the distinct-rank count of one token
    sd = 0.75
    for T, recv in rows:
        n = 8 * T
        assert abs(recv / n - mu) < 5 * sd / math.sqrt(n) + 1e-9, (T, recv)


# --------------------------------------------------------------------------
# Brute force on tiny inputs: the definition enumerated a different way
# --------------------------------------------------------------------------

def brute_force_route(ids, w, E):
    R, T, K = ids.shape
    Epr = E // R
    valid = lambda e: 0 <= e < E
    dests = [[{int(e) // Epr for e in ids[s, t] if valid(e)} for t in range(T)]
             for s in range(R)]
    slot = np.full((R, T, R), -1)
    wd = np.zeros((R, T, R), np.float32)
    for s in range(R):
        for t in range(T):
            for d in dests[s][t]:
                # slot = number of earlier tokens of the same source sent to d
                slot[s, t, d] = sum(1 for u in range(t) if d in dests[s][u])
                acc = F32(0.0)
                for k in range(K):
                    if valid(ids[s, t, k]) and ids[s, t, k] // Epr == d:
                        acc = F32(acc + w[s, t, k])
                wd[s, t, d] = acc
    counts = np.zeros((R, R), int)
    for d in range(R):
        for s in range(R):
            counts[d, s] = sum(1 for t in range(T) if d in dests[s][t])
    local = np.zeros((R, Epr), int)
    for e in ids.ravel():
        if valid(e):
            local[e // Epr, e % Epr] += 1
    bad = sum(1 for e in ids.ravel() if not valid(e) and e != -1)
    return slot, wd, counts, local, bad


@pytest.mark.parametrize("seed", range(4))
def test_route_brute_force(oracle, seed):
    rng = np.random.default_rng(seed)
    R, T, K, E = [(4, 37, 3, 16), (2, 16, 2, 8), (8, 20, 8, 64), (3, 9, 5, 12)][seed]
    ids = rng.integers(-1, E, (R, T, K)).astype(np.int32)   # repeats and -1 allowed
    if seed == 3:
        ids[0, 0, 0] = E          # invalid ids are counted and skipped
        ids[1, 2, 1] = -7
    w = rng.standard_normal((R, T, K)).astype(np.float32)
    m = T + 3
    r = oracle.route(ids, w, E, m)
    slot, wd, counts, local, bad = brute_force_route(ids, w, E)
    assert np.array_equal(r["send_slot"], slot)
    assert np.array_equal(r["wd"].view(np.uint32), wd.view(np.uint32))
    assert np.array_equal(r["recv_counts"], counts)
    assert np.array_equal(r["local_expert_counts"], local)
    assert r["invalid"] == bad
    for d in range(R):
        for s in range(R):
            toks = [t for t in range(T) if slot[s, t, d] >= 0]
            assert list(r["src_token"][d, s, :len(toks)]) == toks
            assert np.all(r["src_token"][d, s, len(toks):] == -1)


def test_route_invariants_decode_shape(oracle):
    from combine_topk_ids_rank_gb300 import synth
    R, T, E, K = 8, 64, 256, 8
    ids = synth.topk_ids(3, R, T, E, K)
    r = oracle.route(ids, synth.topk_weights(3, R, T, K), E, T)
    pop = np.array([bin(int(v)).count("1") for v in r["dmask"].ravel()])
    assert r["recv_counts"].sum() == pop.sum()
    assert r["local_expert_counts"].sum() == (ids >= 0).sum()
    seen = set()
    for d in range(R):
        for s in range(R):
            c = r["recv_counts"][d, s]
            for j in range(c):
                t = r["src_token"][d, s, j]
                assert r["send_slot"][s, t, d] == j
                seen.add((s, t, d))
    assert len(seen) == pop.sum()
    assert np.all((r["send_slot"] >= 0) == (((r["dmask"][..., None] >> np.arange(R)) & 1) == 1))


# --------------------------------------------------------------------------
# Dispatch: identity encoded in the payload, metadata masking
# --------------------------------------------------------------------------

def test_dispatch_payload_identity(oracle):
    R, T, K, E, H = 4, 50, 3, 16, 72     # H not a multiple of 64 nor of 8*32
    rng = np.random.default_rng(7)
    ids = rng.integers(-1, E, (R, T, K)).astype(np.int32)
    w = rng.random((R, T, K)).astype(np.float32)
    m = 64
    # x[s,t,:] encodes (s, t, h) with small integers, exact in bf16
    x = np.empty((R, T, H), np.float32)
    for s in range(R):
        for t in range(T):
            x[s, t] = np.arange(H) % 200
            x[s, t, 0], x[s, t, 1] = s, t
    r = oracle.route(ids, w, E, m)
    pad = np.uint16(0xFFFF)
    d = oracle.dispatch(ids, w, bits(x), E, m, r,
                        recv_x=np.full((R, R, m, H), pad, np.uint16),
                        recv_ids=np.full((R, R, m, K), -99, np.int32),
                        recv_w=np.full((R, R, m, K), -9.0, np.float32))
    Epr = E // R
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            rows = f32(d["recv_x"][dd, s, :c])
            assert np.all(rows[:, 0] == s)
            assert np.array_equal(rows[:, 1].astype(int), r["src_token"][dd, s, :c])
            assert np.all(rows[:, 2:] == (np.arange(2, H) % 200))
            assert np.all(d["recv_x"][dd, s, c:] == pad)          # padding untouched
            assert np.all(d["recv_ids"][dd, s, c:] == -99)
            for j in range(c):
                t = r["src_token"][dd, s, j]
                for k in range(K):
                    e = ids[s, t, k]
                    local = 0 <= e < E and e // Epr == dd
                    assert d["recv_ids"][dd, s, j, k] == (e if local else -1)
                    assert d["recv_w"][dd, s, j, k] == (w[s, t, k] if local else 0.0)


# --------------------------------------------------------------------------
# Combine: closed forms with identity experts, exactly-once reduction
# --------------------------------------------------------------------------

def _identity_case(oracle, R=4, T=40, K=4, E=32, H=64, seed=5, weights=None):
    from combine_topk_ids_rank_gb300 import synth
    ids = synth.topk_ids(seed, R, T, E, K)
    w = synth.topk_weights(seed, R, T, K) if weights is None else weights
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    r = oracle.route(ids, w, E, T)
    d = oracle.dispatch(ids, w, x, E, T, r)
    return ids, w, x, r, d


def test_identity_unweighted_is_n_times_x(oracle):
    ids, w, x, r, d = _identity_case(oracle)
    c = oracle.combine(r, d["recv_x"], weighted=False)
    R, T, H = x.shape
    n = np.array([bin(int(v)).count("1") for v in r["dmask"].ravel()], np.float32)
    # n*x is exact in binary32 (8-bit significand times n <= 8); the result is
    # the round-to-nearest-even of that exact value
    exact = n[:, None] * f32(x).reshape(R * T, H)
    assert np.array_equal(c["acc"], exact)
    assert np.array_equal(c["out"], bits(exact))


def test_identity_weighted_dyadic_returns_x_once(oracle):
    R, T, K = 4, 40, 8
    w = np.full((R, T, K), 1.0 / K, np.float32)       # sums exactly to 1
    ids, w, x, r, d = _identity_case(oracle, R=R, T=T, K=K, weights=w)
    c = oracle.combine(r, d["recv_x"], weighted=True)
    # reduced exactly once: x, not 2x (the double-reduce failure)
    assert np.array_equal(c["out"], x.reshape(R * T, -1))


def test_weighted_sum_within_fp32_error_bound(oracle):
    from combine_topk_ids_rank_gb300 import synth
    R, T, K, E, H = 8, 24, 8, 64, 40
    ids = synth.topk_ids(11, R, T, E, K)
    w = synth.topk_weights(11, R, T, K)
    r = oracle.route(ids, w, E, T)
    eo = synth.expert_out_planes(11, R, T, H, r["recv_counts"])
    c = oracle.combine(r, eo, weighted=True)
    Epr = E // R
    for s in range(R):
        for t in range(T):
            terms, absum = np.zeros(H), np.zeros(H)
            for dd in range(R):
                j = r["send_slot"][s, t, dd]
                if j < 0:
                    continue
                wsum = sum(float(w[s, t, k]) for k in range(K) if ids[s, t, k] // Epr == dd)
                v = f32(eo[dd, s, j]).astype(np.float64)
                terms += wsum * v
                absum += abs(wsum * v)
            got = c["acc"][s * T + t].astype(np.float64)
            # <= 8 fp32 products and adds, plus the fp32 sum of the weights
            assert np.all(np.abs(got - terms) <= 24 * 2.0 ** -24 * absum + 1e-30)


def test_ascending_rank_order_closed_form(oracle):
    # messages 2^24, 1, -2^24 on ranks 0, 1, 2: in fp32, (2^24 + 1) rounds to
    # 2^24 (tie to even), so ascending order gives exactly 0; any other order
    # that adds the 1 after a cancellation gives 1.
    R, E, K, H = 3, 3, 3, 8
    ids = route_to_ranks([[[0, 1, 2]] for _ in range(R)], R, E, K)
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 1)
    vals = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    eo = planes_with(r, R, 1, H, lambda d, s, j: vals[d])
    c = oracle.combine(r, eo, weighted=False)
    assert np.all(c["acc"] == 0.0)


def test_weighted_product_is_not_fused(oracle):
    # rank 0: weight 1, message -(1 + 2^-7); rank 1: weight 1 + 2^-23,
    # message 1 + 2^-7.  Rounded product then add gives 2^-23 exactly; a fused
    # multiply-add keeps the 2^-30 term.  The pages: no FMA in the combine.
    R, E, K, H = 2, 2, 2, 8
    ids = route_to_ranks([[[0, 1]], [[0, 1]]], R, E, K)
    w = np.zeros(ids.shape, np.float32)
    w[:, :, 0] = 1.0
    w[:, :, 1] = np.float32(1 + 2.0 ** -23)
    r = oracle.route(ids, w, E, 1)
    vals = [-(1 + 2.0 ** -7), 1 + 2.0 ** -7]
    eo = planes_with(r, R, 1, H, lambda d, s, j: vals[d])
    c = oracle.combine(r, eo, weighted=True)
    assert np.all(c["acc"] == np.float32(2.0 ** -23))


# --------------------------------------------------------------------------
# Fused epilogue: special cases that reduce to closed forms / a library routine
# --------------------------------------------------------------------------

def test_residual_add_uses_fp32_sum(oracle):
    # acc = 1 + 3*2^-9 (messages 1, 2^-9, 2^-8: exact in fp32), residual -2^-9:
    # the fp32 sum 1 + 2^-8 is exact and a tie, so residual_out = bf16 1.0.
    # Narrowing acc first would give 1.0078125.
    R, E, K, H = 3, 3, 3, 8
    ids = route_to_ranks([[[0, 1, 2]] for _ in range(R)], R, E, K)
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 1)
    vals = [1.0, 2.0 ** -9, 2.0 ** -8]
    eo = planes_with(r, R, 1, H, lambda d, s, j: vals[d])
    res = bits(np.full((R, 1, H), -(2.0 ** -9), np.float32))
    gam = bits(np.ones(H, np.float32))
    c = oracle.combine(r, eo, weighted=False, residual=res, gamma=gam, eps=1e-6)
    assert np.all(f32(c["residual_out"]) == 1.0)


@pytest.mark.parametrize("cval", [1e-3, 0.75, -3.0])
def test_rmsnorm_constant_row_closed_form(oracle, cval):
    # one message per token equal to c everywhere, residual 0: hsum = c, so
    # y = c / sqrt(c^2 + eps) * gamma.
    R, E, K, H, eps = 2, 2, 1, 96, 1e-6
    ids = route_to_ranks([[[0], [1]], [[1], [0]]], R, E, K)
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 2)
    c_bf = float(f32(bits(np.float32(cval))))
    eo = planes_with(r, R, 2, H, lambda d, s, j: c_bf)
    res = np.zeros((R, 2, H), np.uint16)
    g = bits((1.0 + 0.1 * np.sin(np.arange(H))).astype(np.float32))
    out = oracle.combine(r, eo, weighted=False, residual=res, gamma=g, eps=eps)
    eps32 = float(np.float32(eps))          # eps crosses the ABI as binary32
    expect = c_bf / math.sqrt(c_bf * c_bf + eps32) * f32(g).astype(np.float64)
    assert np.allclose(out["y"], expect[None, :], rtol=1e-12, atol=0)


def test_rmsnorm_matches_library_routine(oracle):
    import torch
    from combine_topk_ids_rank_gb300 import synth
    R, T, K, E, H = 4, 12, 4, 16, 200
    ids = synth.topk_ids(2, R, T, E, K)
    w = synth.topk_weights(2, R, T, K)
    r = oracle.route(ids, w, E, T)
    eo = synth.expert_out_planes(2, R, T, H, r["recv_counts"])
    res = synth.per_rank_rows(2, synth.RESIDUAL, R, T, H)
    g = synth.gamma(2, H)
    c = oracle.combine(r, eo, weighted=True, residual=res, gamma=g, eps=1e-6)
    # hsum is the binary32 sum of the reduced row and the residual
    hsum32 = c["acc"] + f32(res).reshape(R * T, H)
    hsum = torch.from_numpy(hsum32.astype(np.float64))
    ref = torch.nn.functional.rms_norm(hsum, (H,), weight=torch.from_numpy(
        f32(g).astype(np.float64)), eps=float(np.float32(1e-6))).numpy()
    assert np.allclose(c["y"], ref, rtol=1e-12, atol=1e-12)
    # out is y narrowed once (through binary32)
    assert np.array_equal(c["out"], bits(c["y"].astype(np.float32)))


def test_tokens_without_experts(oracle):
    R, E, K, H = 2, 4, 2, 16
    ids = np.full((R, 3, K), -1, np.int32)
    ids[0, 1] = [0, 3]
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 3)
    assert r["dmask"][0, 0] == 0 and r["dmask"][1, 2] == 0
    eo = planes_with(r, R, 3, H, lambda d, s, j: 1.0)
    res = bits(np.full((R, 3, H), 0.5, np.float32))
    c0 = oracle.combine(r, eo, weighted=False)
    assert np.all(f32(c0["out"]).reshape(R, 3, H)[1] == 0.0)
    c1 = oracle.combine(r, eo, weighted=False, residual=res,
                        gamma=bits(np.ones(H, np.float32)), eps=0.0)
    # no expert: hsum = residual, y = RMSNorm(residual) = 1 for a constant row
    assert np.all(f32(c1["residual_out"]).reshape(R, 3, H)[1] == 0.5)
    assert np.allclose(c1["y"].reshape(R, 3, H)[1], 1.0)


def test_token_subset_matches_full(oracle):
    from combine_topk_ids_rank_gb300 import synth
    R, T, K, E, H = 4, 20, 4, 16, 48
    ids = synth.topk_ids(9, R, T, E, K)
    w = synth.topk_weights(9, R, T, K)
    r = oracle.route(ids, w, E, T)
    eo = synth.expert_out_planes(9, R, T, H, r["recv_counts"])
    res = synth.per_rank_rows(9, synth.RESIDUAL, R, T, H)
    g = synth.gamma(9, H)
    full = oracle.combine(r, eo, True, res, g, 1e-6)
    pick = np.array([0, 7, 33, R * T - 1])
    sub = oracle.combine(r, eo, True, res, g, 1e-6, tokens=pick)
    for key in ("acc", "out", "residual_out", "y"):
        assert np.array_equal(sub[key], full[key][pick])


# --------------------------------------------------------------------------
# Compatibility reduction: bf16 tree over top-k slots
# --------------------------------------------------------------------------

def test_probe_topk_tree_gives_the_pages_bf16_tree_value(oracle):
    g = read_golden("reduction_discriminator.txt")
    contribs = [float(eval(v, {})) for v in g["contributions"].split(",")]
    R = len(contribs)
    E, K, H = R, R, 8
    ids = route_to_ranks([[list(range(R))] for _ in range(R)], R, E, K)
    r = oracle.route(ids, np.full(ids.shape, 0.125, np.float32), E, 1)
    eo = planes_with(r, R, 1, H, lambda d, s, j: contribs[d])
    c = oracle.combine_topk_tree(r, ids, E, eo)
    assert np.all(f32(c["out"]) == float(g["bf16_tree"]))            # 1.0078125


def test_topk_tree_blanks_duplicate_ranks(oracle):
    g = read_golden("routing_probes.txt")
    R, E, K, H = 2, 4, 2, 8
    ids = np.array([[[0, 1]], [[2, 3]]], np.int32)      # both experts on one rank
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 1)
    eo = planes_with(r, R, 1, H, lambda d, s, j: 1.0)
    c = oracle.combine_topk_tree(r, ids, E, eo)
    assert np.all(f32(c["out"]) == float(g["duplicate_experts_one_rank"]))


def test_topk_tree_keeps_top_k_slot_order(oracle):
    # slots [rank 2: 2^-8, rank 1: 2^-8, rank 0: 1.0, empty]: the tree gives
    # (2^-8 + 2^-8) + (1 + 0) = 1 + 2^-7 exactly; compacting in rank order
    # would give (1 + 2^-8) + 2^-8 -> 1.0 (ties to even twice).
    R, E, K, H = 3, 3, 4, 8
    ids = np.array([[[2, 1, 0, -1]]] * R, np.int32)
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 1)
    vals = [1.0, 2.0 ** -8, 2.0 ** -8]
    eo = planes_with(r, R, 1, H, lambda d, s, j: vals[d])
    c = oracle.combine_topk_tree(r, ids, E, eo)
    assert np.all(f32(c["out"]) == 1.0078125)
    # the fp32 rank-order reduction of the same messages narrows to 1.0078125
    # too (1 + 2^-7 exact); the tree differs from it on the pages' probe above
    full = oracle.combine(r, eo, weighted=False)
    assert np.all(f32(full["out"]) == 1.0078125)


def test_topk_tree_fused_epilogue_matches_rank_sum_when_exact(oracle):
    # with messages whose sums are exact in bf16 the two reductions agree, and
    # so do their fused epilogues
    R, E, K, H = 4, 16, 4, 32
    ids = np.array([[[0, 5, 9, 13]] * 3] * R, np.int32)
    r = oracle.route(ids, np.ones(ids.shape, np.float32), E, 3)
    eo = planes_with(r, R, 3, H, lambda d, s, j: float(d + 1))
    res = bits(np.full((R, 3, H), 0.5, np.float32))
    gam = bits(np.ones(H, np.float32))
    a = oracle.combine_topk_tree(r, ids, E, eo, res, gam, 1e-6)
    b = oracle.combine(r, eo, False, res, gam, 1e-6)
    assert np.array_equal(a["residual_out"], b["residual_out"])
    assert np.array_equal(a["out"], b["out"])


# --------------------------------------------------------------------------
# FP8 (e4m3) payloads: conversion pinned to a library routine, scaling to
# closed forms and the format's error bound
# --------------------------------------------------------------------------

def test_fp8_narrowing_matches_library_routine(oracle):
    import torch
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 60,
                           rng.standard_normal(4000).astype(np.float32) * 1e-2,
                           (rng.random(4000).astype(np.float32) - 0.5) * 2 ** -5,
                           np.array([448, -448, 0, -0.0, 2 ** -9, 2 ** -10, 3 * 2 ** -11,
                                     2 ** -6, 15 * 2 ** -10, 0.5, 0.5625, 0.53125],
                                    np.float32)])
    vals = vals[np.abs(vals) <= 448]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_bits(vals), ref)
    codes = np.arange(256, dtype=np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = oracle.fp8_to_f32(codes)
    assert np.array_equal(np.isnan(got), np.isnan(dec))
    assert np.array_equal(got[~np.isnan(got)], dec[~np.isnan(dec)])


def test_fp8_saturates_and_keeps_nan(oracle):
    codes = oracle.fp8_bits(np.array([449.0, 1e30, -600.0, np.inf, np.nan], np.float32))
    assert list(codes[:4]) == [0x7E, 0x7E, 0xFE, 0x7E]
    assert codes[4] & 0x7F == 0x7F


def test_fp8_row_scaling_closed_forms(oracle):
    # amax 448: scale 1, codes are the plain narrowing; an all-zero row has
    # scale 1 and zero codes; any row's scale is amax / 448 in binary32
    r = np.array([448.0, -3.0, 0.5, 2 ** -9, 0.0, 100.0, -448.0, 7.0], np.float32)
    q, sc = oracle.quantize_rows_fp8(bits(np.stack([r, np.zeros(8, np.float32)])))
    assert sc[0] == 1.0 and np.array_equal(q[0], oracle.fp8_bits(r))
    assert sc[1] == 1.0 and not q[1].any()
    x = bits(np.random.default_rng(6).standard_normal((5, 64)).astype(np.float32))
    q, sc = oracle.quantize_rows_fp8(x)
    amax = np.abs(f32(x)).max(axis=1)
    assert np.array_equal(sc, (amax / np.float32(448)).astype(np.float32))
    assert (np.abs(oracle.fp8_to_f32(q)).max(axis=1) == 448.0).all()


def test_fp8_round_trip_within_format_bound(oracle):
    # e4m3 keeps 3 mantissa bits: a relative half-unit of 2^-4 for normals,
    # an absolute half-unit of 2^-10 (times the scale) for subnormals
    x = bits(np.random.default_rng(7).standard_normal((64, 256)).astype(np.float32) *
             np.logspace(-3, 2, 64, dtype=np.float32)[:, None])
    q, sc = oracle.quantize_rows_fp8(x)
    back = oracle.fp8_to_f32(q) * sc[:, None]
    xv = f32(x)
    assert (np.abs(back - xv) <= 2.0 ** -4 * np.abs(xv) + 2.0 ** -10 * sc[:, None] * 1.0001).all()


# The binary32-row quantiser (the FP8 combine output: the value the bf16
# combine would narrow, quantised per token).  Same format reading as above:
# scale = amax |v| / 448 in binary32, codes = e4m3(RN32(v / scale)).

def test_fp8_f32_rows_closed_forms(oracle):
    # amax exactly 448 -> scale 1 and the plain narrowing of each value (the
    # values are not bf16-representable, so nothing passes through bf16)
    r = np.array([448.0, -3.3, 0.51, 1.1 * 2 ** -9, 0.0, 100.7, -447.9, 7.01], np.float32)
    z = np.zeros(8, np.float32)
    q, sc = oracle.quantize_f32_rows_fp8(np.stack([r, z]))
    assert sc[0] == 1.0 and np.array_equal(q[0], oracle.fp8_bits(r))
    assert sc[1] == 1.0 and not q[1].any()
    # negative-dominated rows: the scale comes from the magnitude of the most
    # negative value; amax 896 gives scale 2 exactly, codes of v / 2
    n = np.array([[-896.0, 3.0, 448.0, -1.0], [5.0, -7.0, 1.0, -0.25]], np.float32)
    q, sc = oracle.quantize_f32_rows_fp8(n)
    assert sc[0] == 2.0
    assert np.array_equal(oracle.fp8_to_f32(q[0]), np.array([-448.0, 1.5, 224.0, -0.5], np.float32))
    assert sc[1] == np.float32(7.0) / np.float32(448.0)
    assert oracle.fp8_to_f32(q[1])[1] == -448.0


def test_fp8_f32_rows_match_library_cast(oracle):
    # random binary32 rows (not bf16-representable, either sign dominant):
    # scale = amax / 448 in binary32 (numpy), codes = torch's e4m3 cast of the
    # binary32 quotient row / scale
    import torch
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((48, 200)) * np.logspace(-6, 6, 48)[:, None]).astype(np.float32)
    x[::3] -= np.float32(3) * np.abs(x[::3]).max(axis=1, keepdims=True)  # negative-dominated
    x[5] = 0.0
    assert (f32(bits(x[:4])) != x[:4]).any()
    q, sc = oracle.quantize_f32_rows_fp8(x)
    amax = np.abs(x).max(axis=1)
    want_sc = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(sc.view(np.uint32), want_sc.view(np.uint32))
    quot = (x / want_sc[:, None]).astype(np.float32)
    assert np.abs(quot).max() <= 448.0 * (1 + 2.0 ** -22)
    ref = torch.from_numpy(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_fp8_f32_rows_round_trip_over_the_binary32_range(oracle):
    # row maxima from 2^-120 to 3e38: dequantised values stay within the
    # format's half step, 2^-4 |x| for normals plus 2^-10 * scale for
    # subnormals (the product taken in float64 so that it adds no rounding)
    rng = np.random.default_rng(9)
    amax = np.exp2(np.linspace(-120.0, np.log2(3e38), 40))
    x = (rng.standard_normal((40, 128)) * (amax / 4.0)[:, None]).astype(np.float32)
    x[:, 0] = amax.astype(np.float32) * np.where(np.arange(40) % 2 == 0, 1, -1)
    q, sc = oracle.quantize_f32_rows_fp8(x)
    back = oracle.fp8_to_f32(q).astype(np.float64) * sc.astype(np.float64)[:, None]
    xv = x.astype(np.float64)
    tol = 2.0 ** -4 * np.abs(xv) * (1 + 2.0 ** -20) + 2.0 ** -10 * sc.astype(np.float64)[:, None]
    assert (np.abs(back - xv) <= tol).all()
    assert np.array_equal(np.abs(oracle.fp8_to_f32(q[:, 0])), np.full(40, 448.0, np.float32))


# --------------------------------------------------------------------------
# Expert-major layout (one expert per received row, "weighted-kernel-sum")
# --------------------------------------------------------------------------

def brute_force_route_experts(ids, w, E, m):
    """The definition enumerated expert by expert: expert e's rows are the
    tokens, in ascending (s, t), whose valid ids contain e."""
    R, T, K = ids.shape
    cap = R * m
    counts = np.zeros(E, np.int32)
    src_row = np.full((E, cap), -1, np.int32)
    send_row = np.full((R, T, K), -1, np.int32)
    wsum = np.zeros((R, T, K), np.float32)
    for e in range(E):
        j = 0
        for s in range(R):
            for t in range(T):
                ks = [k for k in range(K) if ids[s, t, k] == e]
                if not ks:
                    continue
                acc = F32(0.0)
                for k in ks:
                    acc = F32(acc + w[s, t, k])
                send_row[s, t, ks[0]] = e * cap + j
                wsum[s, t, ks[0]] = acc
                src_row[e, j] = s * T + t
                j += 1
        counts[e] = j
    valid = ids[(ids >= 0) & (ids < E)]
    local = np.bincount(valid, minlength=E).astype(np.int32)
    return dict(recv_counts=counts, src_row=src_row, send_row=send_row, wsum=wsum,
                local_expert_counts=local)


@pytest.mark.parametrize("seed", range(3))
def test_route_experts_brute_force(oracle, seed):
    rng = np.random.default_rng(40 + seed)
    R, T, K, E = [(2, 5, 3, 4), (3, 9, 4, 12), (4, 16, 6, 8)][seed]
    m = T + seed
    ids = rng.integers(-1, E, (R, T, K)).astype(np.int32)   # -1 and repeats
    ids[0, 0, :] = -1
    w = rng.random((R, T, K)).astype(np.float32)
    got = oracle.route_experts(ids, w, E, m)
    ref = brute_force_route_experts(ids, w, E, m)
    for key in ("recv_counts", "src_row", "send_row", "local_expert_counts"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(got["wsum"].view(np.uint32), ref["wsum"].view(np.uint32))
    # every (token, distinct valid expert) has exactly one row
    n_pairs = sum(len(set(x for x in ids[s, t] if 0 <= x < E))
                  for s in range(R) for t in range(T))
    assert got["recv_counts"].sum() == n_pairs
    bad = ids.copy()
    bad[1, 2, 0] = E
    assert oracle.route_experts(bad, w, E, m)["invalid"] == 1


def _expert_identity(oracle, ids, w, E, H=32, seed=9):
    """Expert outputs equal to the received rows (identity experts)."""
    R, T, K = ids.shape
    x = bits(np.random.default_rng(seed).standard_normal((R, T, H)).astype(np.float32))
    r = oracle.route_experts(ids, w, E, T)
    eo = oracle.dispatch_experts(x, E, T, r)
    return x, r, eo


def test_expert_dispatch_payload_identity(oracle):
    R, T, K, E = 3, 11, 4, 9
    ids = np.random.default_rng(2).integers(-1, E, (R, T, K)).astype(np.int32)
    w = np.ones((R, T, K), np.float32)
    H = 8
    x = np.zeros((R, T, H), np.uint16)
    for s in range(R):
        for t in range(T):
            x[s, t, :] = bits(np.float32(s * 64 + t))     # the row names its token
    r = oracle.route_experts(ids, w, E, T)
    rx = oracle.dispatch_experts(x, E, T, r)
    for e in range(E):
        for j in range(r["recv_counts"][e]):
            s, t = divmod(int(r["src_row"][e, j]), T)
            assert f32(rx[e, j, 0]) == s * 64 + t and e in ids[s, t]


def test_expert_identity_unweighted_counts_distinct_experts(oracle):
    R, T, K, E = 4, 20, 6, 16
    ids = np.random.default_rng(3).integers(-1, E, (R, T, K)).astype(np.int32)
    w = np.ones((R, T, K), np.float32)
    x, r, eo = _expert_identity(oracle, ids, w, E)
    out = oracle.combine_experts(r, eo, False)["out"].reshape(R, T, -1)
    for s in range(R):
        for t in range(T):
            n = len(set(v for v in ids[s, t] if 0 <= v < E))
            assert np.array_equal(out[s, t], bits(F32(n) * f32(x[s, t])))


def test_expert_identity_weighted_sums_duplicate_weights(oracle):
    # weights 1/8 on every slot, duplicates included: sum_k w_k x = x exactly
    R, T, K, E = 3, 16, 8, 12
    ids = np.random.default_rng(4).integers(0, E, (R, T, K)).astype(np.int32)
    ids[0, 0, :] = 5                                    # all eight slots one expert
    w = np.full((R, T, K), 0.125, np.float32)
    x, r, eo = _expert_identity(oracle, ids, w, E)
    out = oracle.combine_experts(r, eo, True)["out"].reshape(R, T, -1)
    assert np.array_equal(out, x)
    assert r["wsum"][0, 0, 0] == 1.0 and (r["send_row"][0, 0, 1:] == -1).all()


def test_expert_combine_sums_in_problem_order(oracle):
    # top-k order [5, 1, 3] with messages 2^24, 1, -2^24: in problem order
    # (2^24 + 1) rounds to 2^24 and the sum is 0; in expert-id order it is 1
    E, H = 8, 4
    ids = np.array([[[5, 1, 3]]], np.int32)
    w = np.ones((1, 1, 3), np.float32)
    r = oracle.route_experts(ids, w, E, 1)
    eo = np.zeros((E, 1, H), np.uint16)
    for e, v in ((5, 2.0 ** 24), (1, 1.0), (3, -2.0 ** 24)):
        eo[e, 0, :] = bits(np.full(H, v, np.float32))
    out = oracle.combine_experts(r, eo, False)
    assert (out["acc"] == 0.0).all()


def test_expert_combine_fused_matches_rank_layout_when_one_expert_per_rank(oracle):
    # with one expert per rank and the expert outputs equal per rank, the two
    # layouts describe the same sums in the same (ascending) order
    R, T, K, E, H = 4, 12, 4, 4, 16
    ids = np.stack([np.stack([np.random.default_rng(s * 100 + t).permutation(E)[:K]
                              for t in range(T)]) for s in range(R)]).astype(np.int32)
    ids.sort(axis=2)
    w = np.random.default_rng(6).random((R, T, K)).astype(np.float32)
    rng = np.random.default_rng(7)
    res = bits(rng.standard_normal((R, T, H)).astype(np.float32))
    gam = bits(1 + 0.1 * rng.standard_normal(H).astype(np.float32))
    re = oracle.route_experts(ids, w, E, T)
    rr = oracle.route(ids, w, E, T)
    eo_e = np.zeros((E, R * T, H), np.uint16)
    eo_r = np.zeros((R, R, T, H), np.uint16)
    vals = bits(rng.standard_normal((R, T, E, H)).astype(np.float32))
    for s in range(R):
        for t in range(T):
            for k in range(K):
                e = ids[s, t, k]
                eo_e[e, re["send_row"][s, t, k] - e * R * T] = vals[s, t, e]
                eo_r[e, s, rr["send_slot"][s, t, e]] = vals[s, t, e]
    a = oracle.combine_experts(re, eo_e, True, res, gam, 1e-6)
    b = oracle.combine(rr, eo_r, True, res, gam, 1e-6)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["residual_out"], b["residual_out"])


# --------------------------------------------------------------------------
# Expert-side grouped product (the consumer between dispatch and combine)
# --------------------------------------------------------------------------

def test_expert_gemm_identity_and_power_of_two_weights(oracle):
    E, cap, H = 3, 10, 32
    rng = np.random.default_rng(11)
    x = bits(rng.standard_normal((E, cap, H)).astype(np.float32))
    counts = np.array([10, 0, 7], np.int32)
    eye = np.stack([np.eye(H, dtype=np.float32) * (2.0 ** e) for e in range(E)])
    y = oracle.expert_gemm(x, bits(eye), counts)
    for e in range(E):
        assert np.array_equal(y[e, :counts[e]], f32(x[e, :counts[e]]) * 2.0 ** e)
        assert np.isnan(y[e, counts[e]:]).all()          # rows past a count untouched


def test_expert_gemm_matches_library_matmul(oracle):
    # a library routine (numpy's float64 matmul) on a non-square, non-symmetric case
    E, cap, H, N = 4, 9, 24, 40
    rng = np.random.default_rng(12)
    x = bits(rng.standard_normal((E, cap, H)).astype(np.float32))
    w = bits(rng.standard_normal((E, N, H)).astype(np.float32))
    counts = np.array([9, 3, 0, 5], np.int32)
    y = oracle.expert_gemm(x, w, counts)
    for e in range(E):
        c = counts[e]
        ref = f32(x[e, :c]).astype(np.float64) @ f32(w[e]).astype(np.float64).T
        assert np.allclose(y[e, :c], ref, rtol=0, atol=1e-12)


def test_expert_gemm_fp8_identity_and_library_matmul(oracle):
    # identity weights (code 0x38 = 1.0) with unit channel scales give back
    # sx * f(qx); random codes agree with numpy's float64 matmul of the
    # decoded values times the two scales (a library routine)
    E, cap, H = 2, 6, 32
    rng = np.random.default_rng(21)
    qx = rng.integers(0, 256, (E, cap, H)).astype(np.uint8)
    qx[(qx & 0x7F) == 0x7F] = 0x10                      # no NaN codes
    sx = rng.uniform(0.5, 4.0, (E, cap)).astype(np.float32)
    counts = np.array([6, 4], np.int32)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    qw = np.stack([eye, eye])
    y = oracle.expert_gemm_fp8(qx, sx, qw, np.ones((E, H), np.float32), counts)
    fx = oracle.fp8_to_f32(qx).astype(np.float64)
    for e in range(E):
        c = counts[e]
        assert np.array_equal(y[e, :c], fx[e, :c] * sx[e, :c, None].astype(np.float64))
        assert np.isnan(y[e, c:]).all()
    N = 24
    qw = rng.integers(0, 256, (E, N, H)).astype(np.uint8)
    qw[(qw & 0x7F) == 0x7F] = 0x21
    sw = rng.uniform(0.01, 2.0, (E, N)).astype(np.float32)
    y = oracle.expert_gemm_fp8(qx, sx, qw, sw, counts)
    fw = oracle.fp8_to_f32(qw).astype(np.float64)
    for e in range(E):
        c = counts[e]
        ref = (fx[e, :c] @ fw[e].T) * sx[e, :c, None] * sw[e][None, :]
        assert np.allclose(y[e, :c], ref, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# Expert-side product on the rank planes: each received row's local experts,
# their bf16 outputs summed with the gates in ascending k, one narrowing
# --------------------------------------------------------------------------

def _rank_planes(oracle, R=4, T=30, K=4, E=16, H=32, seed=13):
    from combine_topk_ids_rank_gb300 import synth
    ids = synth.topk_ids(seed, R, T, E, K)
    w = synth.topk_weights(seed, R, T, K)
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    r = oracle.route(ids, w, E, T)
    d = oracle.dispatch(ids, w, x, E, T, r)
    return ids, w, x, r, d


def test_expert_gemm_rank_identity_weights_count_local_experts(oracle):
    # W_e = I for every expert, no gates: each row's message is n * x, with n
    # the row's local (valid) ids; n * x is exact in binary32, so the message
    # is torch's round-to-nearest-even of n * x (a library routine)
    import torch
    R, T, K, E, H = 4, 30, 4, 8, 32           # 2 experts per rank: rows carry 1 or 2
    ids, w, x, r, d = _rank_planes(oracle, R, T, K, E, H)
    eye = bits(np.stack([np.eye(H, dtype=np.float32)] * E))
    msg = oracle.expert_gemm_rank(d["recv_x"], d["recv_ids"], d["recv_w"], r["recv_counts"],
                                  eye, apply_gates=False)
    seen = set()
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            n = (d["recv_ids"][dd, s, :c] >= 0).sum(axis=1).astype(np.float32)
            seen.update(n.tolist())
            want = torch.from_numpy(f32(d["recv_x"][dd, s, :c]) * n[:, None]).to(
                torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(msg[dd, s, :c], want)
            assert (msg[dd, s, c:] == 0xFFFF).all()       # rows past a count untouched
    assert {1.0, 2.0} <= seen


def test_expert_gemm_rank_power_of_two_weights_and_dyadic_gates(oracle):
    # W_e = 2^(e mod 3) I and gates 1/8 (exact): message = x * sum over the
    # row's local k of 2^(e_k mod 3) / 8, exact in binary32 and in bf16 range
    R, T, K, E, H = 2, 20, 8, 8, 16
    ids, _, x, r, _ = _rank_planes(oracle, R, T, K, E, H, seed=14)
    w8 = np.full((R, T, K), 0.125, np.float32)
    d = oracle.dispatch(ids, w8, x, E, T, r)
    scale = 2.0 ** (np.arange(E) % 3)
    W = bits(np.stack([np.eye(H, dtype=np.float32) * scale[e] for e in range(E)]))
    msg = oracle.expert_gemm_rank(d["recv_x"], d["recv_ids"], d["recv_w"], r["recv_counts"], W,
                                  apply_gates=True)
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            rid = d["recv_ids"][dd, s, :c]
            f = np.where(rid >= 0, scale[np.maximum(rid, 0)], 0.0).sum(axis=1) / 8.0
            want = f32(d["recv_x"][dd, s, :c]).astype(np.float64) * f[:, None]
            got = f32(msg[dd, s, :c]).astype(np.float64)
            exact = f32(bits(want.astype(np.float32))).astype(np.float64)
            assert np.array_equal(got, exact)


def test_expert_gemm_rank_matches_library_matmul_and_gate_order(oracle):
    # random weights: each local expert's output is numpy's float64 matmul
    # rounded to binary32 then bf16 (torch), the gates applied in binary32 in
    # ascending k, one product and one sum per term, then bf16
    import torch
    R, T, K, E, H, N = 3, 14, 4, 12, 24, 40
    ids, w, x, r, d = _rank_planes(oracle, R, T, K, E, H, seed=15)
    rng = np.random.default_rng(16)
    W = bits((rng.standard_normal((E, N, H)) / 4).astype(np.float32))
    msg, ym, sm = oracle.expert_gemm_rank(d["recv_x"], d["recv_ids"], d["recv_w"],
                                          r["recv_counts"], W, apply_gates=True,
                                          magnitudes=True)

    def to_bf16(v):
        return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).float().numpy()

    Wf = f32(W).astype(np.float64)
    for dd in range(R):
        for s in range(R):
            for j in range(r["recv_counts"][dd, s]):
                xr = f32(d["recv_x"][dd, s, j]).astype(np.float64)
                acc = np.zeros(N, np.float32)
                ymag = np.zeros(N)
                for k in range(K):
                    e = d["recv_ids"][dd, s, j, k]
                    if e < 0:
                        continue
                    y = Wf[e] @ xr
                    g = d["recv_w"][dd, s, j, k]
                    acc = (acc + (np.float32(g) * to_bf16(y.astype(np.float32))).astype(
                        np.float32)).astype(np.float32)
                    ymag += abs(float(g)) * np.abs(y)
                want = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(
                    np.uint16)
                assert np.array_equal(msg[dd, s, j], want)
                assert np.allclose(ym[dd, s, j], ymag, rtol=1e-12, atol=0)
                assert (sm[dd, s, j] >= ym[dd, s, j] * (1 - 1e-12)).all()


def test_expert_gemm_rank_equals_expert_layout_with_one_expert_per_rank(oracle):
    # one expert per rank and distinct ids: every received row carries exactly
    # one local expert, so without gates the rank message is that expert's
    # bf16 output -- the expert-layout product of the same rows
    R, T, K, H, N = 4, 16, 2, 32, 64
    E = R
    ids, w, x, r, d = _rank_planes(oracle, R, T, K, E, H, seed=17)
    rng = np.random.default_rng(18)
    W = bits((rng.standard_normal((E, N, H)) / 4).astype(np.float32))
    msg = oracle.expert_gemm_rank(d["recv_x"], d["recv_ids"], d["recv_w"], r["recv_counts"], W,
                                  apply_gates=False)
    re = oracle.route_experts(ids, w, E, T)
    xe = oracle.dispatch_experts(x, E, T, re)
    y = oracle.expert_gemm(xe, W, re["recv_counts"])
    for e in range(E):
        rows = np.concatenate([msg[e, s, :r["recv_counts"][e, s]] for s in range(R)])
        c = re["recv_counts"][e]
        assert rows.shape[0] == c
        assert np.array_equal(rows, bits(y[e, :c].astype(np.float32)))


def test_expert_gemm_rank_sums_in_top_k_order(oracle):
    # one row with three local experts in top-k order [2, 0, 1] whose outputs
    # are 2^24, 1 and -2^24 (x = ones, W_e = c_e I): in binary32, ascending k
    # gives (2^24 + 1) - 2^24 = 0; expert-id order or descending k give 1
    R, T, K, E, H = 1, 1, 3, 4, 8
    ids = np.array([[[2, 0, 1]]], np.int32)
    w = np.ones((R, T, K), np.float32)
    x = bits(np.ones((R, T, H), np.float32))
    r = oracle.route(ids, w, E, T)
    d = oracle.dispatch(ids, w, x, E, T, r)
    c = {2: 2.0 ** 24, 0: 1.0, 1: -2.0 ** 24, 3: 0.0}
    W = bits(np.stack([np.eye(H, dtype=np.float32) * c[e] for e in range(E)]))
    msg = oracle.expert_gemm_rank(d["recv_x"], d["recv_ids"], d["recv_w"], r["recv_counts"], W,
                                  apply_gates=False)
    assert (f32(msg[0, 0, 0]) == 0.0).all()


# --------------------------------------------------------------------------
# The product on the rank planes with FP8 operands: the FP8 receive rows
# (codes and one scale per row) times FP8 weights (one scale per channel)
# --------------------------------------------------------------------------

def _fp8_rank_planes(oracle, R, T, K, E, H, seed):
    """Rank planes whose rows are the oracle's FP8 quantisation of each
    token, placed at the slots the routing gives (src_token)."""
    ids, w, x, r, d = _rank_planes(oracle, R, T, K, E, H, seed)
    q, sc = oracle.quantize_rows_fp8(x)
    m = T
    qx = np.zeros((R, R, m, H), np.uint8)
    sx = np.zeros((R, R, m), np.float32)
    for dd in range(R):
        for s in range(R):
            for j in range(r["recv_counts"][dd, s]):
                t = r["src_token"][dd, s, j]
                qx[dd, s, j] = q[s, t]
                sx[dd, s, j] = sc[s, t]
    return ids, w, x, r, d, qx, sx


def _bf16_of(v):
    import torch
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_expert_gemm_rank_fp8_identity_codes_count_local_experts(oracle):
    # qw = identity codes (0x38 = 1.0), unit channel scales, no gates: each
    # expert output is bf16(f32(sx * f(qx))) and the message is n times it,
    # n the row's local ids (n * y exact in binary32 for bf16 y, n <= 2)
    R, T, K, E, H = 4, 30, 4, 8, 32
    ids, w, x, r, d, qx, sx = _fp8_rank_planes(oracle, R, T, K, E, H, seed=31)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    msg = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                      np.stack([eye] * E), np.ones((E, H), np.float32),
                                      apply_gates=False)
    fx = oracle.fp8_to_f32(qx).astype(np.float64)
    seen = set()
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            n = (d["recv_ids"][dd, s, :c] >= 0).sum(axis=1).astype(np.float32)
            seen.update(n.tolist())
            y = f32(_bf16_of((fx[dd, s, :c] * sx[dd, s, :c, None]).astype(np.float32)))
            assert np.array_equal(msg[dd, s, :c], _bf16_of(y * n[:, None]))
            assert (msg[dd, s, c:] == 0xFFFF).all()       # rows past a count untouched
    assert {1.0, 2.0} <= seen


def test_expert_gemm_rank_fp8_matches_library_matmul_and_gate_order(oracle):
    # random weight codes and channel scales: each local expert's output is
    # numpy's float64 matmul of the decoded codes (exact: few-bit products,
    # short sums) times sx * sw, rounded to binary32 and bf16; the gates in
    # binary32 in ascending k, one product and one sum per term, then bf16
    R, T, K, E, H, N = 3, 14, 4, 12, 32, 40
    ids, w, x, r, d, qx, sx = _fp8_rank_planes(oracle, R, T, K, E, H, seed=32)
    rng = np.random.default_rng(33)
    qw = rng.integers(0, 256, (E, N, H)).astype(np.uint8)
    qw[(qw & 0x7F) == 0x7F] = 0x21                      # no NaN codes
    sw = rng.uniform(0.01, 2.0, (E, N)).astype(np.float32)
    msg, ym, sm = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"],
                                              r["recv_counts"], qw, sw, apply_gates=True,
                                              magnitudes=True)
    fx = oracle.fp8_to_f32(qx).astype(np.float64)
    fw = oracle.fp8_to_f32(qw).astype(np.float64)
    for dd in range(R):
        for s in range(R):
            for j in range(r["recv_counts"][dd, s]):
                acc = np.zeros(N, np.float32)
                ymag = np.zeros(N)
                for k in range(K):
                    e = d["recv_ids"][dd, s, j, k]
                    if e < 0:
                        continue
                    y = (fw[e] @ fx[dd, s, j]) * (float(sx[dd, s, j]) * sw[e].astype(np.float64))
                    g = d["recv_w"][dd, s, j, k]
                    acc = (acc + (np.float32(g) * f32(_bf16_of(y.astype(np.float32))))
                           .astype(np.float32)).astype(np.float32)
                    ymag += abs(float(g)) * np.abs(y)
                assert np.array_equal(msg[dd, s, j], _bf16_of(acc))
                assert np.allclose(ym[dd, s, j], ymag, rtol=1e-12, atol=0)
                assert (sm[dd, s, j] >= ym[dd, s, j] * (1 - 1e-12)).all()


def test_expert_gemm_rank_fp8_equals_expert_layout_with_one_expert_per_rank(oracle):
    # one expert per rank: each received row carries exactly one local
    # expert, so without gates the message is bf16 of the expert-layout FP8
    # product of the same codes and scales
    R, T, K, H, N = 4, 16, 2, 32, 48
    E = R
    ids, w, x, r, d, qx, sx = _fp8_rank_planes(oracle, R, T, K, E, H, seed=34)
    rng = np.random.default_rng(35)
    qw = rng.integers(0, 256, (E, N, H)).astype(np.uint8)
    qw[(qw & 0x7F) == 0x7F] = 0x13
    sw = rng.uniform(0.1, 1.0, (E, N)).astype(np.float32)
    msg = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                      qw, sw, apply_gates=False)
    cap = R * T
    qe = np.zeros((E, cap, H), np.uint8)
    se = np.zeros((E, cap), np.float32)
    counts = np.zeros(E, np.int32)
    rows = []
    for e in range(E):
        for s in range(R):
            for j in range(r["recv_counts"][e, s]):
                qe[e, counts[e]] = qx[e, s, j]
                se[e, counts[e]] = sx[e, s, j]
                rows.append(msg[e, s, j])
                counts[e] += 1
    y = oracle.expert_gemm_fp8(qe, se, qw, sw, counts)
    want = np.concatenate([_bf16_of(y[e, :counts[e]].astype(np.float32)) for e in range(E)])
    assert np.array_equal(np.stack(rows), want)


def test_expert_gemm_rank_fp8_sums_in_top_k_order(oracle):
    # one row, three local experts in top-k order [2, 0, 1], codes 1.0
    # everywhere on the diagonal and channel scales 2^24, 1, -2^24: ascending k
    # gives (2^24 + 1) - 2^24 = 0 in binary32; other orders give 1
    R, T, K, E, H = 1, 1, 3, 4, 16
    ids = np.array([[[2, 0, 1]]], np.int32)
    w = np.ones((R, T, K), np.float32)
    x = bits(np.ones((R, T, H), np.float32))
    r = oracle.route(ids, w, E, T)
    d = oracle.dispatch(ids, w, x, E, T, r)
    qx = np.full((R, R, T, H), 0x38, np.uint8)
    sx = np.ones((R, R, T), np.float32)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    c = {2: 2.0 ** 24, 0: 1.0, 1: -2.0 ** 24, 3: 0.0}
    sw = np.stack([np.full(H, c[e], np.float32) for e in range(E)])
    msg = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                      np.stack([eye] * E), sw, apply_gates=False)
    assert (f32(msg[0, 0, 0]) == 0.0).all()


def test_expert_gemm_rank_fp8_row_list_matches_full(oracle):
    # the listed-row form computes exactly the listed rows of the full call
    R, T, K, E, H, N = 2, 12, 4, 8, 32, 16
    ids, w, x, r, d, qx, sx = _fp8_rank_planes(oracle, R, T, K, E, H, seed=36)
    rng = np.random.default_rng(37)
    qw = rng.integers(0, 0x70, (E, N, H)).astype(np.uint8)
    sw = rng.uniform(0.1, 1.0, (E, N)).astype(np.float32)
    full = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                       qw, sw)
    flat = [(dd * R + s) * T + j for dd in range(R) for s in range(R)
            for j in range(r["recv_counts"][dd, s])][::3]
    part = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                       qw, sw, rows=np.array(flat, np.int64))
    fm, pm = full.reshape(-1, N), part.reshape(-1, N)
    assert np.array_equal(pm[flat], fm[flat])
    others = np.setdiff1d(np.arange(fm.shape[0]), flat)
    assert (pm[others] == 0xFFFF).all()


def test_expert_gemm_rank_fp8_gate_product_is_not_fused(oracle):
    # two local experts with outputs 1 and 1 + 2^-7 (unit codes, channel
    # scales 1 and 1 + 2^-7), gates 1 and 1 + 2^-23.  Unfused: the product
    # rounds to 1 + 2^-7 + 2^-23, the sum 2 + 2^-7 + 2^-23 is a binary32 tie
    # that goes to 2 + 2^-7, a bf16 tie that goes to 2.  Fused, the sum sits
    # above both ties and the message is 2 + 2^-6.
    R, T, K, E, H = 1, 1, 2, 2, 16
    ids = np.array([[[0, 1]]], np.int32)
    w = np.array([[[1.0, 1.0 + 2.0 ** -23]]], np.float32)
    x = bits(np.ones((R, T, H), np.float32))
    r = oracle.route(ids, w, E, T)
    d = oracle.dispatch(ids, w, x, E, T, r)
    qx = np.full((R, R, T, H), 0x38, np.uint8)
    sx = np.ones((R, R, T), np.float32)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    sw = np.stack([np.ones(H, np.float32), np.full(H, 1.0 + 2.0 ** -7, np.float32)])
    msg = oracle.expert_gemm_rank_fp8(qx, sx, d["recv_ids"], d["recv_w"], r["recv_counts"],
                                      np.stack([eye] * E), sw, apply_gates=True)
    assert (f32(msg[0, 0, 0]) == 2.0).all()
