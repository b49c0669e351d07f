"""Expert-side grouped product on the tensor cores against the oracle.

InferenceX PR #2450, "CollectiveX: add FlashInfer one-sided NVLink EP for the
GB SKUs", "Why": each expert applies its weights to the rows it received,
between dispatch and combine.  The kernel accumulates bf16 products in fp32
in the tensor cores' own order, so against the oracle's double-precision sum
the bound is the bf16 narrowing of the result (half a unit, at most 2^-8
relative: bf16 keeps 8 significant bits)
plus an fp32 accumulation bound H * 2^-23 * sum_h |x_h w_h|.  Identity and
power-of-two weights are exact and are compared bit for bit.
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


def dispatched(R, T, H, E, K, seed, routing="uniform"):
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2A, MOE_LAYOUT_EXPERT
    ids = synth.topk_ids(seed, R, T, E, K, routing)
    w = synth.topk_weights(seed, R, T, K)
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    a.workspace.fill_(parity.POISON)
    view = a.dispatch(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                      parity.to_dev(x, torch.bfloat16))
    r = oracle.route_experts(ids, w, E, T)
    rx = oracle.dispatch_experts(x, E, T, r)
    return a, view, dict(ids=ids, w=w, x=x, r=r, rx=rx)


def weights(seed, E, N, H, scale):
    rng = np.random.default_rng(seed)
    return parity.f32_to_bits((rng.standard_normal((E, N, H), dtype=np.float32) *
                               np.float32(scale)).astype(np.float32))


def check_rows(got, rx, wb, counts, rows):
    """got: bf16 [E, cap, N] (uint16); compare the listed (e, j) rows."""
    E, _, H = wb.shape
    for e in range(E):
        js = [j for j in rows if j < counts[e]]
        if not js:
            continue
        xs = rx[e, js][None]                                   # [1, n, H]
        y = oracle.expert_gemm(xs, wb[e][None], np.array([len(js)], np.int32))[0]
        xa = np.abs(parity.f32(xs[0]).astype(np.float64))
        wa = np.abs(parity.f32(wb[e]).astype(np.float64))
        bound = 2.0 ** -8 * np.abs(y) * 1.0001 + H * 2.0 ** -23 * (xa @ wa.T) + 1e-30
        err = np.abs(parity.f32(got[e, js]).astype(np.float64) - y)
        assert (err <= bound).all(), (e, float(err.max()), float((err / bound).max()))


@pytest.mark.parametrize("R,T,H,E,K,N", [(2, 64, 128, 4, 2, 128), (3, 50, 192, 6, 3, 384),
                                         (4, 100, 256, 8, 4, 512)])
def test_expert_gemm_small(R, T, H, E, K, N):
    # one and several row tiles, 128- and 256-wide column tiles, 2-4 k-blocks
    a, view, d = dispatched(R, T, H, E, K, seed=R * 10 + K)
    cap = view.plane_stride
    wb = weights(7, E, N, H, 1.0 / np.sqrt(H))
    out = torch.full((E, cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm(parity.to_dev(wb, torch.bfloat16), out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0) and a.phase == 1
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    check_rows(got, d["rx"], wb, counts, range(cap))
    for e in range(E):                                         # rows past a count untouched
        assert (got[e, counts[e]:] == 0x7FC0).all()
    a.combine(None, False)


def test_expert_gemm_power_of_two_identity_is_exact():
    # W_e = 2^(e % 3) I: every output row is its input row scaled, bit for bit
    R, T, H, E, K = 4, 90, 256, 8, 3
    a, view, d = dispatched(R, T, H, E, K, seed=3)
    eye = np.stack([np.eye(H, dtype=np.float32) * 2.0 ** (e % 3) for e in range(E)])
    out = a.expert_gemm(parity.to_dev(parity.f32_to_bits(eye), torch.bfloat16))  # payload
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    for e in range(E):
        c = counts[e]
        ref = parity.f32_to_bits(parity.f32(d["rx"][e, :c]) * np.float32(2.0 ** (e % 3)))
        assert np.array_equal(got[e, :c], ref)
    a.combine(None, False)


def test_expert_gemm_feeds_combine():
    # dispatch -> product into the combine payload -> fused weighted combine,
    # with power-of-two identity weights so the oracle's expert outputs are
    # known exactly without the GPU
    R, T, H, E, K = 4, 64, 256, 8, 4
    a, view, d = dispatched(R, T, H, E, K, seed=4)
    eye = np.stack([np.eye(H, dtype=np.float32) * 2.0 ** -(e % 2) for e in range(E)])
    a.expert_gemm(parity.to_dev(parity.f32_to_bits(eye), torch.bfloat16))
    res = synth.per_rank_rows(4, synth.RESIDUAL, R, T, H)
    gam = synth.gamma(4, H)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(out)
    a.combine(None, True, parity.to_dev(res, torch.bfloat16), parity.to_dev(gam, torch.bfloat16),
              1e-6, out, rout)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    eo = d["rx"].copy()
    for e in range(E):
        eo[e] = parity.f32_to_bits(parity.f32(d["rx"][e]) * np.float32(2.0 ** -(e % 2)))
    oc = oracle.combine_experts(d["r"], eo, True, res, gam, 1e-6)
    assert np.array_equal(parity.to_host_u16(rout).reshape(R * T, H), oc["residual_out"])
    err = np.abs(parity.f32(parity.to_host_u16(out).reshape(R * T, H)).astype(np.float64) -
                 oc["y"])
    assert (err <= parity.ABS_TOL).all() and (err <= parity.REL_TOL * np.abs(oc["y"])).all()


def test_expert_gemm_hidden_7168_many_tiles():
    # DeepSeek-size rows: 112 k-blocks, 28 column tiles, 4 row tiles per expert;
    # sampled rows against the oracle (each row is 7168 x 7168 multiply-adds)
    R, T, H, E, K, N = 8, 64, 7168, 8, 8, 7168
    a, view, d = dispatched(R, T, H, E, K, seed=5)
    cap = view.plane_stride
    wb = weights(9, E, N, H, 1.0 / 84.0)
    out = torch.empty((E, cap, N), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm(parity.to_dev(wb, torch.bfloat16), out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    counts = d["r"]["recv_counts"]
    assert (counts == R * T).all()                  # top-8 of 8: every token everywhere
    check_rows(parity.to_host_u16(out), d["rx"], wb, counts, [0, 127, 128, 300, 511])
    a.combine(None, False)


def test_expert_gemm_contract():
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MoeA2AError, MOE_ERR_PHASE,
                                                     MOE_ERR_INVALID_ARG, MOE_FORMAT_FP8_E4M3,
                                                     MOE_LAYOUT_EXPERT)
    R, T, H, E, K = 2, 16, 128, 4, 2
    wt = torch.zeros((E, 128, H), dtype=torch.bfloat16, device="cuda")
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    ids = parity.to_dev(synth.topk_ids(0, R, T, E, K), torch.int32)
    w = parity.to_dev(synth.topk_weights(0, R, T, K), torch.float32)
    x = torch.zeros((R, T, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeA2AError) as ex:          # no dispatch pending
        a.expert_gemm(wt)
    assert ex.value.status == MOE_ERR_PHASE
    a.dispatch(ids, w, x)
    with pytest.raises(MoeA2AError) as ex:          # N != H into the payload
        a.expert_gemm(torch.zeros((E, 256, H), dtype=torch.bfloat16, device="cuda"))
    assert ex.value.status == MOE_ERR_INVALID_ARG
    a.combine(None, False)
    a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    a.dispatch(ids, w, x)
    with pytest.raises(MoeA2AError) as ex:          # e4m3 rows are not a bf16 operand
        a.expert_gemm(wt)
    assert ex.value.status == MOE_ERR_INVALID_ARG
    a.combine(None, False)
    b = MoeA2A(R, T, H, E, K, "cuda")               # rank layout
    b.dispatch(ids, w, x)
    with pytest.raises(MoeA2AError) as ex:
        b.expert_gemm(wt)
    assert ex.value.status == MOE_ERR_INVALID_ARG
    b.combine(None, False)


# --------------------------------------------------------------------------
# FP8 operands: the FP8 receive format (e4m3 rows + per-row scale) against
# e4m3 weights with per-channel scales (tcgen05 .kind::f8f6f4)
# --------------------------------------------------------------------------

def dispatched_fp8(R, T, H, E, K, seed):
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MOE_LAYOUT_EXPERT,
                                                     MOE_FORMAT_FP8_E4M3)
    ids = synth.topk_ids(seed, R, T, E, K)
    w = synth.topk_weights(seed, R, T, K)
    x = synth.per_rank_rows(seed, synth.X, R, T, H)
    a = MoeA2A(R, T, H, E, K, "cuda", layout=MOE_LAYOUT_EXPERT)
    a.workspace.fill_(parity.POISON)
    a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    view = a.dispatch(parity.to_dev(ids, torch.int32), parity.to_dev(w, torch.float32),
                      parity.to_dev(x, torch.bfloat16))
    r = oracle.route_experts(ids, w, E, T)
    q, sc = oracle.quantize_rows_fp8(x)                  # the oracle's own quantisation
    cap = R * T
    qx = np.zeros((E, cap, H), np.uint8)
    sx = np.ones((E, cap), np.float32)
    for e in range(E):
        for j in range(r["recv_counts"][e]):
            s, t = divmod(int(r["src_row"][e, j]), T)
            qx[e, j], sx[e, j] = q[s, t], sc[s, t]
    return a, view, dict(r=r, qx=qx, sx=sx)


def fp8_weights(seed, E, N, H):
    rng = np.random.default_rng(seed)
    qw = rng.integers(0, 256, (E, N, H)).astype(np.uint8)
    qw[(qw & 0x7F) >= 0x70] &= 0x8F                       # keep |w| small, no NaN codes
    sw = rng.uniform(0.5 / np.sqrt(H), 2.0 / np.sqrt(H), (E, N)).astype(np.float32)
    return qw, sw


def check_rows_fp8(got, d, qw, sw, rows):
    E, _, H = qw.shape
    counts = d["r"]["recv_counts"]
    fw_all = oracle.fp8_to_f32(qw).astype(np.float64)
    for e in range(E):
        js = [j for j in rows if j < counts[e]]
        if not js:
            continue
        y = oracle.expert_gemm_fp8(d["qx"][e, js][None], d["sx"][e, js][None], qw[e][None],
                                   sw[e][None], np.array([len(js)], np.int32))[0]
        fx = np.abs(oracle.fp8_to_f32(d["qx"][e, js]).astype(np.float64))
        absum = (fx @ np.abs(fw_all[e]).T) * d["sx"][e, js, None] * sw[e][None, :]
        bound = (2.0 ** -8 + 2.0 ** -22) * np.abs(y) + H * 2.0 ** -23 * absum + 1e-30
        err = np.abs(parity.f32(got[e, js]).astype(np.float64) - y)
        assert (err <= bound).all(), (e, float(err.max()), float((err / bound).max()))


@pytest.mark.parametrize("R,T,H,E,K,N", [(2, 64, 128, 4, 2, 128), (4, 100, 256, 8, 4, 512),
                                         (3, 50, 384, 6, 3, 384)])
def test_expert_gemm_fp8_small(R, T, H, E, K, N):
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=R + N)
    cap = view.plane_stride
    qw, sw = fp8_weights(11, E, N, H)
    out = torch.full((E, cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_fp8(parity.to_dev(qw, torch.uint8), parity.to_dev(sw, torch.float32), out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    check_rows_fp8(got, d, qw, sw, range(cap))
    counts = d["r"]["recv_counts"]
    for e in range(E):
        assert (got[e, counts[e]:] == 0x7FC0).all()
    a.combine(None, False)


def test_expert_gemm_fp8_identity_is_exact():
    # identity codes (0x38 = 1.0), unit channel scales: out = bf16(f(qx) * sx)
    R, T, H, E, K = 4, 70, 256, 8, 3
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=8)
    eye = np.where(np.eye(H, dtype=bool), 0x38, 0).astype(np.uint8)
    qw = np.ascontiguousarray(np.broadcast_to(eye, (E, H, H)))
    out = a.expert_gemm_fp8(parity.to_dev(qw, torch.uint8),
                            torch.ones((E, H), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    got = parity.to_host_u16(out)
    counts = d["r"]["recv_counts"]
    for e in range(E):
        c = counts[e]
        want = oracle.fp8_to_f32(d["qx"][e, :c]) * d["sx"][e, :c, None]   # fp32 product
        assert np.array_equal(got[e, :c], oracle.bf16_bits(want.astype(np.float32)))
    a.combine(None, False)


def test_expert_gemm_fp8_hidden_7168():
    R, T, H, E, K, N = 8, 32, 7168, 8, 8, 7168
    a, view, d = dispatched_fp8(R, T, H, E, K, seed=12)
    cap = view.plane_stride
    qw, sw = fp8_weights(13, E, N, H)
    out = torch.empty((E, cap, N), dtype=torch.bfloat16, device="cuda")
    a.expert_gemm_fp8(parity.to_dev(qw, torch.uint8), parity.to_dev(sw, torch.float32), out)
    torch.cuda.synchronize()
    assert a.get_error() == (0, 0)
    check_rows_fp8(parity.to_host_u16(out), d, qw, sw, [0, 100, 127, 128, 255])
    a.combine(None, False)


def test_expert_gemm_fp8_contract():
    from combine_topk_ids_rank_gb300.moe_a2a import MoeA2AError, MOE_ERR_INVALID_ARG
    a, view, d = dispatched_fp8(2, 16, 128, 4, 2, seed=1)
    w8 = torch.zeros((4, 128, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(MoeA2AError) as ex:          # bf16 product on e4m3 rows
        a.expert_gemm(torch.zeros((4, 128, 128), dtype=torch.bfloat16, device="cuda"))
    assert ex.value.status == MOE_ERR_INVALID_ARG
    a.expert_gemm_fp8(w8, torch.ones((4, 128), dtype=torch.float32, device="cuda"))
    a.combine(None, False)
