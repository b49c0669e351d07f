"""numpy front end of the C oracle (test infrastructure only).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this module.  It marshals numpy arrays into the plain loops of
moe_oracle.c and shares nothing with the CUDA library.  bf16 tensors are
passed as numpy uint16 arrays holding the raw bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib(path: str = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(handle):
    c_int, c_long, c_float = ctypes.c_int, ctypes.c_long, ctypes.c_float
    p = ctypes.c_void_p
    handle.oracle_f32_from_bf16.argtypes = [ctypes.c_uint16]
    handle.oracle_f32_from_bf16.restype = c_float
    handle.oracle_bf16_from_f32.argtypes = [c_float]
    handle.oracle_bf16_from_f32.restype = ctypes.c_uint16
    handle.oracle_route.argtypes = [c_int] * 5 + [p] * 8
    handle.oracle_route.restype = c_long
    handle.oracle_dispatch.argtypes = [c_int] * 6 + [p] * 8
    handle.oracle_dispatch.restype = None
    handle.oracle_combine.argtypes = ([c_int] * 5 + [p] * 6 + [c_float, p, c_long]
                                      + [p] * 4)
    handle.oracle_combine.restype = None
    handle.oracle_combine_topk_tree.argtypes = ([c_int] * 6 + [p] * 5 + [c_float, p, c_long]
                                                + [p] * 3)
    handle.oracle_combine_topk_tree.restype = None
    handle.oracle_route_experts.argtypes = [c_int] * 5 + [p] * 8
    handle.oracle_route_experts.restype = c_long
    handle.oracle_dispatch_experts.argtypes = [c_int] * 4 + [p] * 4
    handle.oracle_dispatch_experts.restype = None
    handle.oracle_combine_experts.argtypes = ([c_int] * 5 + [p] * 5 + [c_float, p, c_long]
                                              + [p] * 4)
    handle.oracle_combine_experts.restype = None
    handle.oracle_expert_gemm.argtypes = [c_int, c_long, c_int, c_int, p, p, p, p]
    handle.oracle_expert_gemm.restype = None
    handle.oracle_expert_gemm_fp8.argtypes = [c_int, c_long, c_int, c_int] + [p] * 6
    handle.oracle_expert_gemm_fp8.restype = None
    handle.oracle_expert_gemm_rank.argtypes = ([c_int] * 5 + [p] * 5 + [c_int, p, c_long]
                                               + [p] * 3)
    handle.oracle_expert_gemm_rank.restype = None
    handle.oracle_expert_gemm_rank_fp8.argtypes = ([c_int] * 5 + [p] * 7 + [c_int, p, c_long]
                                                   + [p] * 3)
    handle.oracle_expert_gemm_rank_fp8.restype = None
    handle.oracle_f32_from_fp8e4m3.argtypes = [ctypes.c_uint8]
    handle.oracle_f32_from_fp8e4m3.restype = c_float
    handle.oracle_fp8e4m3_from_f32.argtypes = [c_float]
    handle.oracle_fp8e4m3_from_f32.restype = ctypes.c_uint8
    handle.oracle_quantize_rows_fp8.argtypes = [c_long, c_int, p, p, p]
    handle.oracle_quantize_rows_fp8.restype = None
    handle.oracle_quantize_f32_rows_fp8.argtypes = [c_long, c_int, p, p, p]
    handle.oracle_quantize_f32_rows_fp8.restype = None
    return handle


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _need(a, dtype, shape=None):
    a = np.ascontiguousarray(a, dtype=dtype)
    if shape is not None and a.shape != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), a.shape))
    return a


def bf16_bits(values, handle=None):
    """Round binary32 values to bf16 bit patterns with the oracle's rule."""
    h = handle or lib()
    flat = np.asarray(values, dtype=np.float32).ravel()
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = h.oracle_bf16_from_f32(float(v))
    return out.reshape(np.shape(values))


def bf16_to_f32(bits):
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def route(topk_ids, topk_w, num_experts: int, m: int, handle=None):
    """Routing, dedup and slot assignment.  topk_ids/topk_w: [R, T, K]."""
    h = handle or lib()
    ids = _need(topk_ids, np.int32)
    R, T, K = ids.shape
    w = _need(topk_w, np.float32, ids.shape)
    if num_experts % R:
        raise ValueError("num_experts must be a multiple of ep_size")
    if T > m:
        raise ValueError("T > m")
    out = dict(
        dmask=np.empty((R, T), np.uint32),
        wd=np.empty((R, T, R), np.float32),
        send_slot=np.empty((R, T, R), np.int32),
        recv_counts=np.empty((R, R), np.int32),
        src_token=np.empty((R, R, m), np.int32),
        local_expert_counts=np.empty((R, num_experts // R), np.int32),
    )
    out["invalid"] = h.oracle_route(
        R, T, K, num_experts, m, _ptr(ids), _ptr(w), _ptr(out["dmask"]),
        _ptr(out["wd"]), _ptr(out["send_slot"]), _ptr(out["recv_counts"]),
        _ptr(out["src_token"]), _ptr(out["local_expert_counts"]))
    return out


def dispatch(topk_ids, topk_w, x, num_experts: int, m: int, routing,
             recv_x=None, recv_ids=None, recv_w=None, handle=None):
    """Copy rows and masked metadata into padded planes [R, R, m, ...].

    Slots past each plane's count are left as they were in the given (or
    freshly allocated, uninitialised) output arrays."""
    h = handle or lib()
    ids = _need(topk_ids, np.int32)
    R, T, K = ids.shape
    w = _need(topk_w, np.float32, ids.shape)
    xb = _need(x, np.uint16)
    H = xb.shape[-1]
    if xb.shape != (R, T, H):
        raise ValueError("x must be [R, T, H]")
    if recv_x is None:
        recv_x = np.empty((R, R, m, H), np.uint16)
    if recv_ids is None:
        recv_ids = np.empty((R, R, m, K), np.int32)
    if recv_w is None:
        recv_w = np.empty((R, R, m, K), np.float32)
    h.oracle_dispatch(R, T, K, num_experts, H, m, _ptr(ids), _ptr(w), _ptr(xb),
                      _ptr(_need(routing["recv_counts"], np.int32)),
                      _ptr(_need(routing["src_token"], np.int32)),
                      _ptr(recv_x), _ptr(recv_ids), _ptr(recv_w))
    return dict(recv_x=recv_x, recv_ids=recv_ids, recv_w=recv_w)


def combine(routing, expert_out, weighted: bool, residual=None, gamma=None,
            eps: float = 1e-6, tokens=None, handle=None, outputs=None):
    """Reduce each token's per-rank messages once; optional fused epilogue.

    expert_out: uint16 [R, R, m, H] (only valid slots are read).
    residual: uint16 [R, T, H] or None; gamma: uint16 [H] (fused only).
    tokens: optional flat token indices s*T+t; outputs are [ntok, H].
    Returns dict(acc=float32, out=uint16, residual_out=uint16|None, y=float64).
    `outputs` may hold preallocated arrays of those names and shapes.
    """
    h = handle or lib()
    dmask = _need(routing["dmask"], np.uint32)
    R, T = dmask.shape
    eo = expert_out if (isinstance(expert_out, np.ndarray)
                        and expert_out.dtype == np.uint16
                        and expert_out.flags.c_contiguous) else _need(expert_out, np.uint16)
    if eo.ndim != 4 or eo.shape[:2] != (R, R):
        raise ValueError("expert_out must be [R, R, m, H]")
    m, H = eo.shape[2], eo.shape[3]
    tok = None if tokens is None else _need(tokens, np.int64)
    n = R * T if tok is None else tok.shape[0]
    res = None
    gam = None
    if residual is not None:
        res = _need(residual, np.uint16, (R, T, H))
        gam = _need(gamma, np.uint16, (H,))
    o = outputs or {}
    acc = o.get("acc")
    acc = np.empty((n, H), np.float32) if acc is None else acc
    out = o.get("out")
    out = np.empty((n, H), np.uint16) if out is None else out
    rout = None
    if res is not None:
        rout = o.get("residual_out")
        rout = np.empty((n, H), np.uint16) if rout is None else rout
    y = o.get("y")
    y = np.empty((n, H), np.float64) if y is None else y
    for name, a, dt in (("acc", acc, np.float32), ("out", out, np.uint16),
                        ("y", y, np.float64), ("residual_out", rout, np.uint16)):
        if a is not None and (a.shape != (n, H) or a.dtype != dt or not a.flags.c_contiguous):
            raise ValueError("output %s must be a contiguous %s [%d, %d]" % (name, dt, n, H))
    h.oracle_combine(R, T, H, m, int(bool(weighted)), _ptr(dmask),
                     _ptr(_need(routing["send_slot"], np.int32)),
                     _ptr(_need(routing["wd"], np.float32)), _ptr(eo),
                     _ptr(res), _ptr(gam), float(eps), _ptr(tok), n,
                     _ptr(acc), _ptr(out), _ptr(rout), _ptr(y))
    return dict(acc=acc, out=out, residual_out=rout, y=y)


def combine_topk_tree(routing, topk_ids, num_experts: int, expert_out, residual=None,
                      gamma=None, eps: float = 1e-6, tokens=None, handle=None):
    """The bf16 top-k-slot tree reduction (compatibility mode), unweighted.

    Returns dict(out=uint16, residual_out=uint16|None, y=float64), rows per
    requested token."""
    h = handle or lib()
    ids = _need(topk_ids, np.int32)
    R, T, K = ids.shape
    eo = _need(expert_out, np.uint16)
    m, H = eo.shape[2], eo.shape[3]
    tok = None if tokens is None else _need(tokens, np.int64)
    n = R * T if tok is None else tok.shape[0]
    res = gam = rout = None
    if residual is not None:
        res = _need(residual, np.uint16, (R, T, H))
        gam = _need(gamma, np.uint16, (H,))
        rout = np.empty((n, H), np.uint16)
    out = np.empty((n, H), np.uint16)
    y = np.empty((n, H), np.float64)
    h.oracle_combine_topk_tree(R, T, K, num_experts, H, m, _ptr(ids),
                               _ptr(_need(routing["send_slot"], np.int32)), _ptr(eo),
                               _ptr(res), _ptr(gam), float(eps), _ptr(tok), n,
                               _ptr(out), _ptr(rout), _ptr(y))
    return dict(out=out, residual_out=rout, y=y)


def route_experts(topk_ids, topk_w, num_experts: int, m: int, handle=None):
    """Routing of the expert-major layout (one row per distinct (token,
    expert), planes of cap = R * m rows, ascending (source, token)).
    topk_ids/topk_w: [R, T, K]."""
    h = handle or lib()
    ids = _need(topk_ids, np.int32)
    R, T, K = ids.shape
    w = _need(topk_w, np.float32, ids.shape)
    if T > m:
        raise ValueError("T > m")
    E, cap = num_experts, R * m
    out = dict(
        send_row=np.empty((R, T, K), np.int32),
        wsum=np.empty((R, T, K), np.float32),
        recv_counts=np.empty(E, np.int32),
        src_row=np.empty((E, cap), np.int32),
        recv_w=np.empty((E, cap), np.float32),
        local_expert_counts=np.empty(E, np.int32),
        cap=cap,
    )
    out["invalid"] = h.oracle_route_experts(
        R, T, K, E, m, _ptr(ids), _ptr(w), _ptr(out["send_row"]), _ptr(out["wsum"]),
        _ptr(out["recv_counts"]), _ptr(out["src_row"]), _ptr(out["recv_w"]),
        _ptr(out["local_expert_counts"]))
    return out


def dispatch_experts(x, num_experts: int, m: int, routing, recv_x=None, handle=None):
    """recv_x [E, cap, H] (uint16 bf16 bits) of the expert-major layout; rows
    past each count are left as given (zeros if recv_x is None)."""
    h = handle or lib()
    xb = _need(x, np.uint16)
    R, T, H = xb.shape
    cap = R * m
    if recv_x is None:
        recv_x = np.zeros((num_experts, cap, H), np.uint16)
    h.oracle_dispatch_experts(R, num_experts, H, m, _ptr(xb),
                              _ptr(_need(routing["recv_counts"], np.int32)),
                              _ptr(_need(routing["src_row"], np.int32)), _ptr(recv_x))
    return recv_x


def combine_experts(routing, expert_out, weighted: bool, residual=None, gamma=None,
                    eps: float = 1e-6, tokens=None, handle=None):
    """Weighted-kernel-sum combine of the expert-major layout (ascending k).
    expert_out: [E, cap, H] uint16.  Returns dict(acc, out, residual_out, y)
    with one row per requested token."""
    h = handle or lib()
    send_row = _need(routing["send_row"], np.int32)
    R, T, K = send_row.shape
    eo = _need(expert_out, np.uint16)
    H = eo.shape[-1]
    tok = None if tokens is None else _need(tokens, np.int64)
    n = R * T if tok is None else tok.shape[0]
    res = gam = rout = None
    if residual is not None:
        res = _need(residual, np.uint16, (R, T, H))
        gam = _need(gamma, np.uint16, (H,))
        rout = np.empty((n, H), np.uint16)
    acc = np.empty((n, H), np.float32)
    out = np.empty((n, H), np.uint16)
    y = np.empty((n, H), np.float64)
    h.oracle_combine_experts(R, T, K, H, int(bool(weighted)), _ptr(send_row),
                             _ptr(_need(routing["wsum"], np.float32)), _ptr(eo), _ptr(res),
                             _ptr(gam), float(eps), _ptr(tok), n, _ptr(acc), _ptr(out),
                             _ptr(rout), _ptr(y))
    return dict(acc=acc, out=out, residual_out=rout, y=y)


def expert_gemm(x, w, recv_counts, handle=None):
    """Per-expert product y[e][j] = x[e][j] . w[e]^T in double for the rows
    j < recv_counts[e].  x: [E, cap, H] uint16 (bf16 bits), w: [E, N, H]
    uint16.  Returns float64 [E, cap, N] with NaN in the rows past a count."""
    h = handle or lib()
    xb = _need(x, np.uint16)
    wb = _need(w, np.uint16)
    E, cap, H = xb.shape
    N = wb.shape[1]
    if wb.shape != (E, N, H):
        raise ValueError("w must be [E, N, H]")
    y = np.full((E, cap, N), np.nan, np.float64)
    h.oracle_expert_gemm(E, cap, H, N, _ptr(_need(recv_counts, np.int32, (E,))), _ptr(xb),
                         _ptr(wb), _ptr(y))
    return y


def expert_gemm_rank(recv_x, recv_ids, recv_w, recv_counts, w, apply_gates=True, rows=None,
                     magnitudes=False, handle=None):
    """The expert product on the rank planes: for every received row (or the
    flat rows (d*R+s)*m+j listed in `rows`), msg = bf16 of the gate-weighted
    (or plain) binary32 sum, ascending k, of the bf16 outputs of the row's
    local experts.  recv_x [R, R, m, H] uint16, recv_ids [R, R, m, K] int32,
    recv_w [R, R, m, K] float32, recv_counts [R, R], w [E, N, H] uint16.
    Returns msg uint16 [R, R, m, N] (0xFFFF in rows not computed) and, with
    magnitudes=True, also ymag and smag float64 of the same shape."""
    h = handle or lib()
    xb = _need(recv_x, np.uint16)
    R, R2, m, H = xb.shape
    ids = _need(recv_ids, np.int32)
    K = ids.shape[-1]
    if R2 != R or ids.shape != (R, R, m, K):
        raise ValueError("recv_ids must be [R, R, m, K]")
    wb = _need(w, np.uint16)
    N = wb.shape[1]
    if wb.shape[2] != H:
        raise ValueError("w must be [E, N, H]")
    rl = None if rows is None else _need(rows, np.int64)
    msg = np.full((R, R, m, N), 0xFFFF, np.uint16)
    ym = np.full((R, R, m, N), np.nan, np.float64) if magnitudes else None
    sm = np.full((R, R, m, N), np.nan, np.float64) if magnitudes else None
    h.oracle_expert_gemm_rank(R, m, K, H, N, _ptr(_need(recv_counts, np.int32, (R, R))), _ptr(xb),
                              _ptr(ids), _ptr(_need(recv_w, np.float32, ids.shape)), _ptr(wb),
                              int(bool(apply_gates)), _ptr(rl), 0 if rl is None else rl.shape[0],
                              _ptr(msg), _ptr(ym), _ptr(sm))
    return (msg, ym, sm) if magnitudes else msg


def expert_gemm_fp8(qx, sx, qw, sw, recv_counts, handle=None):
    """FP8 operands: y[e][j][n] = sx[e][j] sw[e][n] sum_h f(qx) f(qw) in
    double.  qx [E, cap, H] / qw [E, N, H] uint8 e4m3 codes, sx [E, cap] /
    sw [E, N] float32.  Returns float64 [E, cap, N], NaN past a count."""
    h = handle or lib()
    qxb = _need(qx, np.uint8)
    qwb = _need(qw, np.uint8)
    E, cap, H = qxb.shape
    N = qwb.shape[1]
    if qwb.shape != (E, N, H):
        raise ValueError("qw must be [E, N, H]")
    y = np.full((E, cap, N), np.nan, np.float64)
    h.oracle_expert_gemm_fp8(E, cap, H, N, _ptr(_need(recv_counts, np.int32, (E,))), _ptr(qxb),
                             _ptr(_need(sx, np.float32, (E, cap))), _ptr(qwb),
                             _ptr(_need(sw, np.float32, (E, N))), _ptr(y))
    return y


def expert_gemm_rank_fp8(recv_x8, recv_scale, recv_ids, recv_w, recv_counts, qw, sw,
                         apply_gates=True, rows=None, magnitudes=False, handle=None):
    """The rank-plane product on FP8 operands (oracle_expert_gemm_rank_fp8):
    recv_x8 [R, R, m, H] uint8 e4m3 codes with recv_scale [R, R, m] float32,
    recv_ids [R, R, m, K] int32, recv_w [R, R, m, K] float32, recv_counts
    [R, R], qw [E, N, H] uint8 codes with sw [E, N] float32.  Returns msg
    uint16 [R, R, m, N] (0xFFFF in rows not computed) and, with
    magnitudes=True, also ymag and smag float64 of the same shape."""
    h = handle or lib()
    xb = _need(recv_x8, np.uint8)
    R, R2, m, H = xb.shape
    ids = _need(recv_ids, np.int32)
    K = ids.shape[-1]
    if R2 != R or ids.shape != (R, R, m, K):
        raise ValueError("recv_ids must be [R, R, m, K]")
    wb = _need(qw, np.uint8)
    E, N = wb.shape[0], wb.shape[1]
    if wb.shape[2] != H:
        raise ValueError("qw must be [E, N, H]")
    rl = None if rows is None else _need(rows, np.int64)
    msg = np.full((R, R, m, N), 0xFFFF, np.uint16)
    ym = np.full((R, R, m, N), np.nan, np.float64) if magnitudes else None
    sm = np.full((R, R, m, N), np.nan, np.float64) if magnitudes else None
    h.oracle_expert_gemm_rank_fp8(R, m, K, H, N, _ptr(_need(recv_counts, np.int32, (R, R))),
                                  _ptr(xb), _ptr(_need(recv_scale, np.float32, (R, R, m))),
                                  _ptr(ids), _ptr(_need(recv_w, np.float32, ids.shape)),
                                  _ptr(wb), _ptr(_need(sw, np.float32, (E, N))),
                                  int(bool(apply_gates)), _ptr(rl),
                                  0 if rl is None else rl.shape[0], _ptr(msg), _ptr(ym), _ptr(sm))
    return (msg, ym, sm) if magnitudes else msg


def fp8_bits(values, handle=None):
    """binary32 values -> e4m3 codes (uint8), the oracle's narrowing."""
    h = handle or lib()
    flat = np.asarray(values, dtype=np.float32).ravel()
    out = np.array([h.oracle_fp8e4m3_from_f32(float(v)) for v in flat], np.uint8)
    return out.reshape(np.shape(values))


def fp8_to_f32(codes, handle=None):
    """e4m3 codes -> float32 through the oracle's decoding of all 256 codes."""
    h = handle or lib()
    table = np.array([h.oracle_f32_from_fp8e4m3(c) for c in range(256)], np.float32)
    return table[np.asarray(codes, dtype=np.uint8)]


def quantize_rows_fp8(x_bf16, handle=None):
    """bf16 rows [..., H] -> (e4m3 codes [..., H], fp32 scales [...])."""
    h = handle or lib()
    xb = _need(x_bf16, np.uint16)
    H = xb.shape[-1]
    n = xb.size // H
    q = np.empty(xb.shape, np.uint8)
    sc = np.empty(xb.shape[:-1], np.float32)
    h.oracle_quantize_rows_fp8(n, H, _ptr(xb), _ptr(q), _ptr(sc))
    return q, sc


def quantize_f32_rows_fp8(x_f32, handle=None):
    """binary32 rows [..., H] -> (e4m3 codes, fp32 scales)."""
    h = handle or lib()
    xf = _need(x_f32, np.float32)
    H = xf.shape[-1]
    n = xf.size // H
    q = np.empty(xf.shape, np.uint8)
    sc = np.empty(xf.shape[:-1], np.float32)
    h.oracle_quantize_f32_rows_fp8(n, H, _ptr(xf), _ptr(q), _ptr(sc))
    return q, sc

