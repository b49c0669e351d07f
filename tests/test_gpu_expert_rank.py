"""Expert-side product on the rank planes (moe_expert_gemm_rank, and
moe_expert_gemm_rank_fp8 on the FP8 receive rows) against the oracle,
through the C ABI.

InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided NVLink EP for the
GB SKUs", "Why": each expert applies its weights to the rows it received;
vLLM applies the gates in the MoE layer.  A received row carries the token's
experts that live on its rank; the message is bf16 of the gated fp32 sum, in
ascending top-k order, of the experts' bf16 outputs.

The tensor cores accumulate in their own order, so an expert output may land
one bf16 unit away from the oracle's (exact sum rounded to binary32, then
bf16): at most 2^-7 |y| (bf16 keeps 8 significant bits) plus the fp32
accumulation bound H 2^-23 sum_h |x w|.  Summed with the gates and narrowed
once more, the message may differ by
  2^-7 |msg| + 1.01 (2^-7 + K 2^-23) sum_k |g_k y_k| + 1.01 H 2^-23 sum_k |g_k| sum_h |x w|,
with the two magnitude sums taken from the oracle.  The mean error must also
stay below 2^-8 of the mean message.  Power-of-two diagonal weights and
dyadic gates make every step exact: those cases are compared bit for bit,
and through the whole step (dispatch, product, unweighted fused combine).
On FP8 operands each expert output also carries two fp32 scale multiplies
(2^-22 relative); identity codes with power-of-two channel scales make that
case exact too.
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


def dispatched(R, T, H, E, K, seed, routing="uniform", gates=None):
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A
    ids = synth.topk_ids(seed, R, T, E, K, routing)
    w = synth.topk_weights(seed, R, T, K) if gates is None else gates
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    a = MoeA2A(R, T, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)
    view = a.dispatch(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                      parity.to_dev(x, torch.bfloat16))
    r = oracle.route(ids, w, E, T)
    od = oracle.dispatch(ids, w, x, E, T, r)
    return a, view, dict(ids=ids, w=w, x=x, r=r, od=od)


def weights(seed, E, N, H, scale):
    """bf16 [E, N, H] on the device from torch's seeded normal generator (an
    input of the call, like the routing; up to 26 GB at E = 256, H = N = 7168)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w = torch.empty((E, N, H), dtype=torch.bfloat16, device="cuda")
    for e in range(E):
        w[e] = (torch.randn((N, H), generator=g, device="cuda") * scale).to(torch.bfloat16)
    return w


def valid_rows(counts, m):
    R = counts.shape[0]
    return np.array([(d * R + s) * m + j for d in range(R) for s in range(R)
                     for j in range(counts[d, s])], np.int64)


def check(got, d, w_dev, apply_gates, rows):
    """got: uint16 [R, R, m, N]; compare the listed flat rows with the oracle,
    which receives the weights of the experts those rows carry."""
    od, r = d["od"], d["r"]
    K = od["recv_ids"].shape[-1]
    H = od["recv_x"].shape[-1]
    ids = od["recv_ids"]
    used = np.unique(ids.reshape(-1, K)[rows])
    used = used[used >= 0]
    lut = np.full(w_dev.shape[0], -1, np.int32)
    lut[used] = np.arange(used.size, dtype=np.int32)
    ok = (ids >= 0) & (ids < w_dev.shape[0])    # (padding slots hold anything)
    ids_sub = np.where(ok, lut[np.where(ok, ids, 0)], -1).astype(np.int32)
    wb = parity.to_host_u16(w_dev[torch.from_numpy(used).cuda()].contiguous())
    msg, ym, sm = oracle.expert_gemm_rank(od["recv_x"], ids_sub, od["recv_w"],
                                          r["recv_counts"], wb, apply_gates, rows=rows,
                                          magnitudes=True)
    N = msg.shape[-1]
    g = parity.f32(got.reshape(-1, N)[rows]).astype(np.float64)
    o = parity.f32(msg.reshape(-1, N)[rows]).astype(np.float64)
    ym = ym.reshape(-1, N)[rows]
    sm = sm.reshape(-1, N)[rows]
    bound = (2.0 ** -7 * np.abs(o) + 1.01 * (2.0 ** -7 + K * 2.0 ** -23) * ym +
             1.01 * H * 2.0 ** -23 * sm + 1e-30)
    err = np.abs(g - o)
    assert np.isfinite(g).all()
    assert (err <= bound).all(), (float(err.max()), float((err / bound).max()))
    assert err.mean() <= 2.0 ** -8 * np.abs(o).mean()
    return float(err.max()), float((err == 0).mean())


@pytest.mark.parametrize("R,T,H,E,K,N,gates", [(2, 64, 128, 4, 2, 128, True),
                                               (3, 50, 192, 6, 3, 384, False),
                                               (4, 100, 256, 16, 4, 512, True),
                                               (4, 300, 256, 8, 8, 256, True),
                                               (4, 300, 256, 4, 2, 256, True),
                                               (4, 300, 256, 4, 2, 256, False)])
def test_expert_gemm_rank_small(R, T, H, E, K, N, gates):
    # one and several row tiles per expert, 128- and 256-wide column tiles,
    # rows carrying one to K local experts (with one expert per rank every
    # row carries one: its message comes straight from the product's
    # epilogue), every row compared
    a, view, d = dispatched(R, T, H, E, K, seed=R * 10 + K)
    m = view.plane_stride
    wb = weights(7, E, N, H, 1.0 / np.sqrt(H))
    out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_rank(wb, gates, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 1
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    check(got, d, wb, gates, valid_rows(counts, m))
    for dd in range(R):                       # rows past a count are not written
        for s in range(R):
            assert np.isnan(parity.f32(got[dd, s, counts[dd, s]:])).all()
    a.combine(None, False)


def test_expert_gemm_rank_exact_weights_bit_exact_and_whole_step():
    # W_e = 2^(e mod 3) I and gates 1/8: every expert output, gated sum and
    # the unweighted fused combine are exact or correctly rounded once, so
    # the GPU equals the oracle bit for bit through dispatch, product and
    # combine (the product writing the combine payload)
    R, T, H, E, K = 8, 64, 256, 64, 8
    gates = np.full((R, T, K), 0.125, np.float32)
    a, view, d = dispatched(R, T, H, E, K, seed=3, gates=gates)
    scale = 2.0 ** (np.arange(E) % 3)
    wb = parity.f32_to_bits(np.stack([np.eye(H, dtype=np.float32) * scale[e]
                                      for e in range(E)]))
    a.expert_gemm_rank(parity.to_dev(wb, torch.bfloat16), True)      # into the payload
    torch.cuda.synchronize()
    got = parity.to_host_u16(a.combine_payload())
    od, r = d["od"], d["r"]
    msg = oracle.expert_gemm_rank(od["recv_x"], od["recv_ids"], od["recv_w"],
                                  r["recv_counts"], wb, True)
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            assert np.array_equal(got[dd, s, :c], msg[dd, s, :c]), (dd, s)
    res = synth.per_rank_rows(3, synth.RESIDUAL, R, T, H)
    gam = synth.gamma(3, H)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    a.combine(None, False, parity.to_dev(res, torch.bfloat16), parity.to_dev(gam, torch.bfloat16),
              1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    oc = oracle.combine(r, msg, False, res, gam, 1e-6)
    assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"])
    y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
    err = np.abs(y - oc["y"])
    assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()


def test_expert_gemm_rank_decode_shape():
    # decode: 8 ranks x 64 tokens, H = N = 7168, 256 experts, top-8, output
    # into the combine payload; a seeded sample of rows (plus a few planes'
    # first and last rows) against the oracle, every row checked as written
    R, T, H, E, K = 8, 64, 7168, 256, 8
    a, view, d = dispatched(R, T, H, E, K, seed=0)
    m = view.plane_stride
    wb = weights(11, E, H, H, 1.0 / np.sqrt(H))
    a.expert_gemm_rank(wb, True)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(a.combine_payload())
    counts = d["r"]["recv_counts"]
    rows = valid_rows(counts, m)
    assert np.isfinite(parity.f32(got.reshape(-1, H)[rows])).all()
    rng = np.random.default_rng(1)
    pick = set(rng.choice(rows, 24, replace=False).tolist())
    for dd, s in ((0, 0), (3, 5), (7, 7)):     # a few planes' first and last rows
        c = counts[dd, s]
        if c:
            pick.update([(dd * R + s) * m, (dd * R + s) * m + c - 1])
    check(got, d, wb, True, np.array(sorted(pick), np.int64))
    a.combine(None, False)


def test_expert_gemm_rank_prefill_shape():
    # prefill-sized rank planes: 8 ranks x 4096 tokens, H = 7168, 256 experts,
    # top-8 with Zipf(1.2) popularity (expert 0 in almost every token: one
    # expert with hundreds of row tiles), N = 256 into a caller buffer
    R, T, H, E, K, N = 8, 4096, 7168, 256, 8, 256
    a, view, d = dispatched(R, T, H, E, K, seed=0, routing="zipf")
    m = view.plane_stride
    wb = weights(12, E, N, H, 1.0 / np.sqrt(H))
    out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_rank(wb, True, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    rows = valid_rows(counts, m)
    assert np.isfinite(parity.f32(got.reshape(-1, N)[rows])).all()
    rng = np.random.default_rng(2)
    pick = set(rng.choice(rows, 512, replace=False).tolist())
    for dd in range(R):
        for s in range(R):
            c = counts[dd, s]
            if c:
                pick.update([(dd * R + s) * m, (dd * R + s) * m + c - 1])
    check(got, d, wb, True, np.array(sorted(pick), np.int64))
    for dd in range(R):
        for s in range(R):
            assert np.isnan(parity.f32(got[dd, s, counts[dd, s]:])).all()
    a.combine(None, False)


def test_expert_gemm_rank_repeat_calls_bit_identical():
    # the pairs' order inside an expert list is not fixed, the results are
    R, T, H, E, K, N = 4, 200, 256, 8, 4, 256
    a, view, d = dispatched(R, T, H, E, K, seed=9)
    m = view.plane_stride
    wb = weights(13, E, N, H, 1.0 / np.sqrt(H))
    outs = []
    for _ in range(3):
        out = torch.zeros((R, R, m, N), dtype=torch.bfloat16, device="cuda")
        a.expert_gemm_rank(wb, True, out)
        outs.append(parity.to_host_u16(out))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    a.combine(None, False)


def test_expert_gemm_rank_contract():
    from combine_topk_ids_rank_gb300 import moe_a2a as mod
    R, T, H, E, K = 2, 16, 128, 4, 2
    a = mod.MoeA2A(R, T, H, E, K, "cuda")
    wb = torch.zeros((E, H, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mod.MoeA2AError) as e:          # no dispatch pending
        a.expert_gemm_rank(wb, True)
    assert e.value.status == mod.MOE_ERR_PHASE
    a2, view, d = dispatched(R, T, H, E, K, seed=1)
    need = mod.moe_expert_gemm_rank_scratch_bytes(a2.cfg, H)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mod.MoeA2AError) as e:
        a2.expert_gemm_rank(wb, True, scratch=small)
    assert e.value.status == mod.MOE_ERR_CAPACITY
    assert a2.phase == 1
    a2.combine(None, False)


# --------------------------------------------------------------------------
# FP8 operands (moe_expert_gemm_rank_fp8): the FP8 receive rows (e4m3 codes,
# one scale per received row) against e4m3 weights with one scale per
# output channel.  Beyond the bf16 bound, the epilogue's two fp32 scale
# multiplies add at most 2^-22 |y_k| per expert output.
# --------------------------------------------------------------------------

def dispatched_fp8(R, T, H, E, K, seed, routing="uniform", gates=None):
    """A rank-layout dispatch in the FP8 receive format, and the oracle's
    rank planes: its routing, its quantisation of every token placed at the
    slots of that routing (codes qx [R, R, m, H], scales sx [R, R, m])."""
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    ids = synth.topk_ids(seed, R, T, E, K, routing)
    w = synth.topk_weights(seed, R, T, K) if gates is None else gates
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    a = MoeA2A(R, T, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)
    a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    view = a.dispatch(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                      parity.to_dev(x, torch.bfloat16))
    m = view.plane_stride
    r = oracle.route(ids, w, E, T)
    od = oracle.dispatch(ids, w, x, E, T, r)
    q, sc = oracle.quantize_rows_fp8(x)
    qx = np.zeros((R, R, m, H), np.uint8)
    sx = np.zeros((R, R, m), np.float32)
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            src = r["src_token"][dd, s, :c]
            qx[dd, s, :c] = q[s, src]
            sx[dd, s, :c] = sc[s, src]
    return a, view, dict(ids=ids, w=w, x=x, r=r, od=od, qx=qx, sx=sx)


def fp8_weights(seed, E, N, H):
    """e4m3 codes [E, N, H] (no NaN codes, |w| <= 1.875 before the scale)
    from torch's seeded generator on the device, and channel scales [E, N]
    near 1 / sqrt(H)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    qw = torch.randint(0, 256, (E, N, H), dtype=torch.uint8, device="cuda", generator=g)
    big = (qw & 0x7F) >= 0x40
    qw = torch.where(big, qw & 0xBF, qw)                # exponent field below 8: |f| < 2
    sw = (torch.rand((E, N), generator=g, device="cuda") * 1.5 + 0.5) / np.sqrt(H)
    return qw.contiguous(), sw.float().contiguous()


def check_fp8(got, d, qw_dev, sw_dev, apply_gates, rows):
    """As check(), through oracle.expert_gemm_rank_fp8 on the oracle's codes."""
    od, r = d["od"], d["r"]
    K = od["recv_ids"].shape[-1]
    H = d["qx"].shape[-1]
    ids = od["recv_ids"]
    used = np.unique(ids.reshape(-1, K)[rows])
    used = used[used >= 0]
    lut = np.full(qw_dev.shape[0], -1, np.int32)
    lut[used] = np.arange(used.size, dtype=np.int32)
    ok = (ids >= 0) & (ids < qw_dev.shape[0])
    ids_sub = np.where(ok, lut[np.where(ok, ids, 0)], -1).astype(np.int32)
    sel = torch.from_numpy(used).cuda()
    qw = qw_dev[sel].cpu().numpy()
    sw = sw_dev[sel].cpu().numpy()
    msg, ym, sm = oracle.expert_gemm_rank_fp8(d["qx"], d["sx"], ids_sub, od["recv_w"],
                                              r["recv_counts"], qw, sw, apply_gates,
                                              rows=rows, magnitudes=True)
    N = msg.shape[-1]
    g = parity.f32(got.reshape(-1, N)[rows]).astype(np.float64)
    o = parity.f32(msg.reshape(-1, N)[rows]).astype(np.float64)
    ym = ym.reshape(-1, N)[rows]
    sm = sm.reshape(-1, N)[rows]
    bound = (2.0 ** -7 * np.abs(o) + 1.01 * (2.0 ** -7 + 2.0 ** -22 + K * 2.0 ** -23) * ym +
             1.01 * H * 2.0 ** -23 * sm + 1e-30)
    err = np.abs(g - o)
    assert np.isfinite(g).all()
    assert (err <= bound).all(), (float(err.max()), float((err / bound).max()))
    assert err.mean() <= 2.0 ** -8 * np.abs(o).mean()
    return float(err.max()), float((err == 0).mean())


@pytest.mark.parametrize("R,T,H,E,K,N,gates", [(2, 64, 128, 4, 2, 128, True),
                                               (3, 50, 384, 6, 3, 384, False),
                                               (4, 100, 256, 16, 4, 512, True),
                                               (4, 300, 256, 8, 8, 256, True),
                                               (4, 300, 256, 4, 2, 256, True),
                                               (4, 300, 128, 4, 2, 128, False)])
def test_expert_gemm_rank_fp8_small(R, T, H, E, K, N, gates):
    # one and several row tiles per expert, 128- and 256-wide column tiles,
    # rows carrying one (written by the product's epilogue) to K local
    # experts (summed after it), every row compared
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=R * 10 + K + 1)
    m = view.plane_stride
    qw, sw = fp8_weights(7, E, N, H)
    out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_rank_fp8(qw, sw, gates, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 1
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    check_fp8(got, d, qw, sw, gates, valid_rows(counts, m))
    for dd in range(R):                       # rows past a count are not written
        for s in range(R):
            assert np.isnan(parity.f32(got[dd, s, counts[dd, s]:])).all()
    a.combine(None, False)


def test_expert_gemm_rank_fp8_exact_weights_bit_exact_and_whole_step():
    # identity codes (1.0) with channel scales 2^(e mod 3) and gates 1/8: an
    # expert output is bf16(f32(sx f(qx)) 2^j) on both sides (one product on
    # the tensor cores, exact), so messages and the unweighted fused combine
    # after them equal the oracle bit for bit
    R, T, H, E, K = 8, 64, 256, 64, 8
    gates = np.full((R, T, K), 0.125, np.float32)
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=4, gates=gates)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    qw = np.ascontiguousarray(np.broadcast_to(eye, (E, H, H)))
    sw = np.repeat((2.0 ** (np.arange(E) % 3)).astype(np.float32)[:, None], H, axis=1)
    a.expert_gemm_rank_fp8(parity.to_dev(qw, torch.uint8), parity.to_dev(sw, torch.float32),
                           True)                                   # into the payload
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(a.combine_payload())
    od, r = d["od"], d["r"]
    msg = oracle.expert_gemm_rank_fp8(d["qx"], d["sx"], od["recv_ids"], od["recv_w"],
                                      r["recv_counts"], qw, sw, True)
    for dd in range(R):
        for s in range(R):
            c = r["recv_counts"][dd, s]
            assert np.array_equal(got[dd, s, :c], msg[dd, s, :c]), (dd, s)
    res = synth.per_rank_rows(4, synth.RESIDUAL, R, T, H)
    gam = synth.gamma(4, H)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    a.combine(None, False, parity.to_dev(res, torch.bfloat16), parity.to_dev(gam, torch.bfloat16),
              1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    oc = oracle.combine(r, msg, False, res, gam, 1e-6)
    assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"])
    y = parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64)
    err = np.abs(y - oc["y"])
    assert ((err <= parity.ABS_TOL) & (err <= parity.REL_TOL * np.abs(oc["y"]))).all()


def test_expert_gemm_rank_fp8_decode_shape():
    # decode: 8 ranks x 64 tokens, H = N = 7168, 256 experts, top-8, output
    # into the combine payload; a seeded sample of rows against the oracle
    R, T, H, E, K = 8, 64, 7168, 256, 8
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=0)
    m = view.plane_stride
    qw, sw = fp8_weights(11, E, H, H)
    a.expert_gemm_rank_fp8(qw, sw, True)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(a.combine_payload())
    counts = d["r"]["recv_counts"]
    rows = valid_rows(counts, m)
    assert np.isfinite(parity.f32(got.reshape(-1, H)[rows])).all()
    rng = np.random.default_rng(3)
    pick = set(rng.choice(rows, 10, replace=False).tolist())
    c = counts[7, 7]
    if c:
        pick.update([(7 * R + 7) * m, (7 * R + 7) * m + c - 1])
    check_fp8(got, d, qw, sw, True, np.array(sorted(pick), np.int64))
    a.combine(None, False)


def test_expert_gemm_rank_fp8_prefill_shape():
    # prefill-sized rank planes: 8 ranks x 4096 tokens, H = 7168, 256
    # experts, top-8 with Zipf(1.2) popularity, N = 256 into a caller buffer
    R, T, H, E, K, N = 8, 4096, 7168, 256, 8, 256
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=0, routing="zipf")
    m = view.plane_stride
    qw, sw = fp8_weights(12, E, N, H)
    out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_rank_fp8(qw, sw, True, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    rows = valid_rows(counts, m)
    assert np.isfinite(parity.f32(got.reshape(-1, N)[rows])).all()
    rng = np.random.default_rng(4)
    pick = set(rng.choice(rows, 384, replace=False).tolist())
    for dd in range(R):
        for s in range(R):
            c = counts[dd, s]
            if c:
                pick.update([(dd * R + s) * m, (dd * R + s) * m + c - 1])
    check_fp8(got, d, qw, sw, True, np.array(sorted(pick), np.int64))
    for dd in range(R):
        for s in range(R):
            assert np.isnan(parity.f32(got[dd, s, counts[dd, s]:])).all()
    a.combine(None, False)


def test_expert_gemm_rank_fp8_repeat_calls_bit_identical():
    R, T, H, E, K, N = 4, 200, 256, 8, 4, 256
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=9)
    m = view.plane_stride
    qw, sw = fp8_weights(13, E, N, H)
    outs = []
    for _ in range(3):
        out = torch.zeros((R, R, m, N), dtype=torch.bfloat16, device="cuda")
        a.expert_gemm_rank_fp8(qw, sw, True, out)
        outs.append(parity.to_host_u16(out))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    a.combine(None, False)


def test_expert_gemm_rank_fp8_contract():
    from combine_topk_ids_rank_gb300 import moe_a2a as mod
    R, T, H, E, K = 2, 16, 128, 4, 2
    qw = torch.zeros((E, H, H), dtype=torch.uint8, device="cuda")
    sw = torch.ones((E, H), dtype=torch.float32, device="cuda")
    wb = torch.zeros((E, H, H), dtype=torch.bfloat16, device="cuda")
    a, view, d = dispatched(R, T, H, E, K, seed=1)             # bf16 receive format
    with pytest.raises(mod.MoeA2AError) as e:
        a.expert_gemm_rank_fp8(qw, sw, True)
    assert e.value.status == mod.MOE_ERR_INVALID_ARG
    a.combine(None, False)
    b, view, d = dispatched_fp8(R, T, H, E, K, seed=1)         # FP8 receive format
    with pytest.raises(mod.MoeA2AError) as e:                 # bf16 product on e4m3 rows
        b.expert_gemm_rank(wb, True)
    assert e.value.status == mod.MOE_ERR_INVALID_ARG
    scratch = torch.empty(mod.moe_expert_gemm_rank_scratch_bytes(b.cfg, H), dtype=torch.uint8,
                          device="cuda")
    st = mod.moe_expert_gemm_rank_fp8(b.handle, qw.data_ptr(), 0, H, 1, 0,   # no channel scales
                                      scratch.data_ptr(), scratch.numel())
    assert st == mod.MOE_ERR_INVALID_ARG
    with pytest.raises(mod.MoeA2AError) as e:                 # scratch too small
        b.expert_gemm_rank_fp8(qw, sw, True, scratch=scratch[:-256])
    assert e.value.status == mod.MOE_ERR_CAPACITY
    b.expert_gemm_rank_fp8(qw, sw, True)
    torch.cuda.synchronize()
    assert b.get_error() == (0, 0) and b.phase == 1
    b.combine(None, False)


@pytest.mark.parametrize("fp8", [False, True])
def test_expert_gemm_rank_varlen_and_dead_ranks(fp8):
    # per-rank token counts and two dead ranks: the product sees exactly the
    # rows and local experts of the oracle's routing on the masked ids (a
    # token past its rank's count, or an expert on a dead rank, is absent)
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    R, M, H, E, K, N = 8, 96, 256, 64, 8, 256
    counts = [96, 0, 50, 1, 96, 33, 70, 5]
    dead = (2, 5)
    ids = synth.topk_ids(21, R, M, E, K)
    w = synth.topk_weights(21, R, M, K)
    x = synth.per_rank_rows(21, synth.X, R, M, H)
    mids = ids.copy()
    for s, c in enumerate(counts):
        mids[s, c:] = -1
    for dd in dead:
        mids[(mids >= 0) & (mids // (E // R) == dd)] = -1
    a = MoeA2A(R, M, H, E, K, "cuda")
    a.workspace.fill_(parity.POISON)
    if fp8:
        a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    a.set_active_ranks(0xFF & ~sum(1 << dd for dd in dead))
    view = a.dispatch_varlen(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                             parity.to_dev(x, torch.bfloat16), counts)
    assert view.plane_stride == M
    r = oracle.route(mids, w, E, M)
    assert np.array_equal(view.recv_counts.cpu().numpy(), r["recv_counts"])
    od = oracle.dispatch(mids, w, x, E, M, r)
    d = dict(r=r, od=od)
    out = torch.full((R, R, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if fp8:
        q, sc = oracle.quantize_rows_fp8(x)
        d["qx"] = np.zeros((R, R, M, H), np.uint8)
        d["sx"] = np.zeros((R, R, M), np.float32)
        for dd in range(R):
            for s in range(R):
                c = r["recv_counts"][dd, s]
                d["qx"][dd, s, :c] = q[s, r["src_token"][dd, s, :c]]
                d["sx"][dd, s, :c] = sc[s, r["src_token"][dd, s, :c]]
        qw, sw = fp8_weights(22, E, N, H)
        a.expert_gemm_rank_fp8(qw, sw, True, out)
    else:
        wb = weights(22, E, N, H, 1.0 / np.sqrt(H))
        a.expert_gemm_rank(wb, True, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    rows = valid_rows(r["recv_counts"], M)
    if fp8:
        check_fp8(got, d, qw, sw, True, rows)
    else:
        check(got, d, wb, True, rows)
    for dd in range(R):
        for s in range(R):
            assert np.isnan(parity.f32(got[dd, s, r["recv_counts"][dd, s]:])).all()
    assert r["recv_counts"][list(dead)].sum() == 0
    a.combine(None, False)


@pytest.mark.parametrize("fp8", [False, True])
def test_expert_gemm_rank_empty_and_no_pairs(fp8):
    # an empty dispatch, and one whose tokens name no expert (all ids -1):
    # the product queues nothing or finds no pairs, writes nothing and
    # reports no error
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_FORMAT_FP8_E4M3
    R, H, E, K, N = 4, 128, 8, 2, 128
    for T in (0, 20):
        a = MoeA2A(R, 32, H, E, K, "cuda")
        if fp8:
            a.set_recv_format(MOE_FORMAT_FP8_E4M3)
        ids = torch.full((R, T, K), -1, dtype=torch.int32, device="cuda")
        w = torch.ones((R, T, K), dtype=torch.float32, device="cuda")
        x = torch.ones((R, T, H), dtype=torch.bfloat16, device="cuda")
        view = a.dispatch(ids, w, x, 8 if T == 0 else None)
        assert int(view.recv_counts.sum().item()) == 0
        m = view.plane_stride
        out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        if fp8:
            a.expert_gemm_rank_fp8(torch.zeros((E, N, H), dtype=torch.uint8, device="cuda"),
                                   torch.ones((E, N), dtype=torch.float32, device="cuda"),
                                   True, out)
        else:
            a.expert_gemm_rank(torch.zeros((E, N, H), dtype=torch.bfloat16, device="cuda"),
                               True, out)
        torch.cuda.synchronize()
        assert a.get_error() == (0, 0) and a.phase == 1
        assert torch.isnan(out.float()).all()
        a.combine(None, False)


@pytest.mark.parametrize("fp8", [False, True])
def test_expert_gemm_rank_single_rank_top1(fp8):
    # one rank, top-1: every received row carries exactly one local expert,
    # so every message comes from the product's epilogue (bf16(+0 + g y))
    R, T, H, E, K, N = 1, 200, 256, 4, 1, 256
    if fp8:
        a, view, d = dispatched_fp8(R, T, H, E, K, seed=51)
        qw, sw = fp8_weights(52, E, N, H)
    else:
        a, view, d = dispatched(R, T, H, E, K, seed=51)
        wb = weights(52, E, N, H, 1.0 / np.sqrt(H))
    m = view.plane_stride
    out = torch.full((R, R, m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if fp8:
        a.expert_gemm_rank_fp8(qw, sw, True, out)
    else:
        a.expert_gemm_rank(wb, True, out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    rows = valid_rows(d["r"]["recv_counts"], m)
    assert rows.size == T
    if fp8:
        check_fp8(got, d, qw, sw, True, rows)
    else:
        check(got, d, wb, True, rows)
    a.combine(None, False)
