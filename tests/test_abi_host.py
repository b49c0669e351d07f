"""C-ABI contract checks that need no GPU.

The library must load, export every entry point include/moe_a2a.h declares,
and enforce the phase contract and the size/pointer checks on the host
before anything is queued (InferenceX PR #2450, "CollectiveX: add FlashInfer
one-sided NVLink EP for the GB SKUs", "The adapter" table).
"""
import os
import re

import numpy as np
import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_a2a.h")


@pytest.fixture(scope="module")
def abi():
    from combine_topk_ids_rank_gb300 import build_lib
    build_lib.build()
    from combine_topk_ids_rank_gb300 import moe_a2a
    return moe_a2a


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def declared_enum():
    text = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"\b(MOE_\w+)\s*=\s*(\d+)", text)}


def test_exports_every_declared_symbol(abi):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(abi._lib, n), n
    assert set(names) == set(abi.EXPORTS)


def test_status_codes_match_header(abi):
    enum = declared_enum()
    for k, v in enum.items():
        assert getattr(abi, k) == v
    for v in enum.values():
        assert abi.status_string(v) not in ("", "unknown status")


CFG = (8, 4096, 7168, 256, 8)


def test_workspace_bytes_rejects_bad_configs(abi):
    good = abi.moe_a2a_workspace_bytes(abi.config(*CFG))
    # two bf16 payload regions dominate: 2 * R*R*M*H*2 bytes
    assert good >= 2 * 8 * 8 * 4096 * 7168 * 2
    assert good < 2 * 8 * 8 * 4096 * 7168 * 2 * 1.05
    bad = [(0, 4096, 7168, 256, 8), (33, 64, 128, 33 * 2, 2), (8, 0, 7168, 256, 8),
           (8, 64, 7170, 256, 8), (8, 64, 32768, 256, 8), (8, 64, 128, 250, 8),
           (8, 64, 128, 256, 0), (8, 64, 128, 256, 33), (8, 64, 128, 16384, 2)]
    for c in bad:
        assert abi.moe_a2a_workspace_bytes(abi.config(*c)) == 0, c


def test_workspace_sized_once_grows_with_max_tokens(abi):
    a = abi.moe_a2a_workspace_bytes(abi.config(8, 64, 7168, 256, 8))
    b = abi.moe_a2a_workspace_bytes(abi.config(8, 8192, 7168, 256, 8))
    assert b > 100 * a


def _handle(abi, cfg=CFG, nbytes=None):
    c = abi.config(*cfg)
    need = abi.moe_a2a_workspace_bytes(c)
    st, h = abi.moe_a2a_create(c, 1 << 30, need if nbytes is None else nbytes)
    return st, h


def test_create_checks(abi):
    c = abi.config(*CFG)
    need = abi.moe_a2a_workspace_bytes(c)
    assert abi.moe_a2a_create(c, 0, need)[0] == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_create(c, (1 << 30) + 16, need)[0] == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_create(c, 1 << 30, need - 1)[0] == abi.MOE_ERR_CAPACITY
    assert abi.moe_a2a_create(abi.config(0, 1, 8, 1, 1), 1 << 30, need)[0] == \
        abi.MOE_ERR_INVALID_ARG
    st, h = _handle(abi)
    assert st == abi.MOE_OK and abi.moe_a2a_phase(h) == 0
    assert abi.moe_combine_payload(h) >= (1 << 30)
    assert abi.moe_a2a_destroy(h) == abi.MOE_OK


def test_combine_without_dispatch_is_a_phase_error(abi):
    st, h = _handle(abi)
    assert abi.moe_combine(h, 0, 1, 0, 0, 1e-6, 1 << 20, 0, 0) == abi.MOE_ERR_PHASE
    assert abi.moe_a2a_phase(h) == 0
    abi.moe_a2a_destroy(h)


def test_dispatch_capacity_and_argument_checks(abi):
    st, h = _handle(abi)
    A = 1 << 20                       # an aligned stand-in pointer (never touched)
    d = lambda ids, w, x, T, m: abi.moe_dispatch(h, ids, w, x, T, m, 0)[0]
    assert d(A, A, A, 10, 4097) == abi.MOE_ERR_CAPACITY          # runtime max > max
    assert d(A, A, A, 17, 16) == abi.MOE_ERR_CAPACITY            # T > runtime max
    assert d(A, A, A, -1, 16) == abi.MOE_ERR_INVALID_ARG
    assert d(A, A, A, 1, 0) == abi.MOE_ERR_INVALID_ARG
    assert d(0, A, A, 4, 16) == abi.MOE_ERR_INVALID_ARG
    assert d(A, 0, A, 4, 16) == abi.MOE_ERR_INVALID_ARG
    assert d(A, A, 0, 4, 16) == abi.MOE_ERR_INVALID_ARG
    assert d(A, A, A + 8, 4, 16) == abi.MOE_ERR_INVALID_ARG       # x not 16-byte aligned
    assert d(A + 2, A, A, 4, 16) == abi.MOE_ERR_INVALID_ARG       # ids not 4-byte aligned
    assert abi.moe_a2a_phase(h) == 0                              # errors leave the phase
    abi.moe_a2a_destroy(h)


def test_null_handle(abi):
    assert abi.moe_a2a_destroy(None) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_phase(None) == -1
    assert abi.moe_combine_payload(None) == 0
    assert abi.moe_dispatch(None, 0, 0, 0, 0, 1, 0)[0] == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_combine(None, 0, 0, 0, 0, 0.0, 0, 0, 0) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_get_error(None)[0] == abi.MOE_ERR_INVALID_ARG


def test_get_error_before_any_work(abi):
    st, h = _handle(abi)
    assert abi.moe_a2a_get_error(h) == (abi.MOE_OK, 0)
    abi.moe_a2a_destroy(h)


def test_set_reduction_checks(abi):
    st, h = _handle(abi)                      # top_k = 8
    assert abi.moe_a2a_set_reduction(h, abi.MOE_REDUCE_BF16_TOPK_TREE) == abi.MOE_OK
    assert abi.moe_a2a_set_reduction(h, abi.MOE_REDUCE_FP32_RANK_ORDER) == abi.MOE_OK
    assert abi.moe_a2a_set_reduction(h, 7) == abi.MOE_ERR_INVALID_ARG
    abi.moe_a2a_destroy(h)
    st, h = _handle(abi, cfg=(8, 64, 128, 256, 9))
    assert abi.moe_a2a_set_reduction(h, abi.MOE_REDUCE_BF16_TOPK_TREE) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_set_reduction(None, 0) == abi.MOE_ERR_INVALID_ARG
    abi.moe_a2a_destroy(h)


def test_varlen_and_active_rank_checks(abi):
    import ctypes
    st, h = _handle(abi, cfg=(4, 64, 128, 16, 2))
    A = 1 << 20
    d = lambda counts, m: abi.moe_dispatch_varlen(h, A, A, A, counts, m, 0)[0]
    assert d([1, 2, 3, 65], 64) == abi.MOE_ERR_CAPACITY        # a count above runtime max
    assert d([1, -2, 3, 4], 64) == abi.MOE_ERR_INVALID_ARG
    assert d([1, 2, 3, 4], 65) == abi.MOE_ERR_CAPACITY        # runtime max above max
    assert d([1, 2, 3, 4], 0) == abi.MOE_ERR_INVALID_ARG
    assert abi._lib.moe_dispatch_varlen(h, None, None, None, None, 8, None, None) == \
        abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_phase(h) == 0
    assert abi.moe_a2a_set_active_ranks(h, 0b1011) == abi.MOE_OK
    assert abi.moe_a2a_set_active_ranks(h, 0b10000) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_set_active_ranks(None, 1) == abi.MOE_ERR_INVALID_ARG
    abi.moe_a2a_destroy(h)


def test_recv_format_and_fp8_combine_checks(abi):
    st, h = _handle(abi, cfg=(4, 64, 136, 16, 2))     # H = 136: not a multiple of 16
    assert abi.moe_a2a_set_recv_format(h, abi.MOE_FORMAT_FP8_E4M3) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_set_recv_format(h, abi.MOE_FORMAT_BF16) == abi.MOE_OK
    abi.moe_a2a_destroy(h)
    st, h = _handle(abi, cfg=(4, 64, 128, 16, 2))
    assert abi.moe_a2a_set_recv_format(h, abi.MOE_FORMAT_FP8_E4M3) == abi.MOE_OK
    assert abi.moe_a2a_set_recv_format(h, 2) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_set_recv_format(None, 0) == abi.MOE_ERR_INVALID_ARG
    A = 1 << 20
    assert abi.moe_combine_fp8(h, 0, 0, 0, 0, 1e-6, A, A, 0) == abi.MOE_ERR_PHASE
    assert abi.moe_combine_fp8(None, 0, 0, 0, 0, 1e-6, A, A, 0) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_phase(h) == 0
    abi.moe_a2a_destroy(h)


def test_view_struct_matches_header(abi):
    import ctypes
    text = open(HEADER).read()
    body = text[text.index("typedef struct moe_dispatch_view {"):text.index("} moe_dispatch_view_t;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\*?\s*(\w+);", body)
    assert names == [f[0] for f in abi.MoeDispatchView._fields_]


def test_quantize_rows_fp8_checks(abi):
    A = 1 << 20
    q = abi.moe_quantize_rows_fp8
    assert q(A, 0, 64, A, A) == abi.MOE_OK                  # nothing to do, nothing queued
    assert q(A, -1, 64, A, A) == abi.MOE_ERR_INVALID_ARG
    assert q(A, 4, 60, A, A) == abi.MOE_ERR_INVALID_ARG      # H not a multiple of 8
    assert q(A, 4, 32768, A, A) == abi.MOE_ERR_INVALID_ARG
    assert q(0, 4, 64, A, A) == abi.MOE_ERR_INVALID_ARG
    assert q(A + 4, 4, 64, A, A) == abi.MOE_ERR_INVALID_ARG  # x not 16-byte aligned
    assert q(A, 4, 64, A + 8, A) == abi.MOE_ERR_INVALID_ARG
    assert q(A, 4, 64, A, A + 2) == abi.MOE_ERR_INVALID_ARG


def test_expert_layout_host_checks(abi):
    c = abi.config(8, 64, 7168, 256, 8)
    rank = abi.moe_a2a_workspace_bytes_layout(c, abi.MOE_LAYOUT_RANK)
    assert rank == abi.moe_a2a_workspace_bytes(c)
    ex = abi.moe_a2a_workspace_bytes_layout(c, abi.MOE_LAYOUT_EXPERT)
    # two bf16 regions of E * R * M rows dominate
    assert 2 * 256 * 8 * 64 * 7168 * 2 <= ex < 2 * 256 * 8 * 64 * 7168 * 2 * 1.05
    assert abi.moe_a2a_workspace_bytes_layout(c, 2) == 0
    assert abi.moe_a2a_workspace_bytes_layout(abi.config(8, 64, 128, 2048, 8),
                                              abi.MOE_LAYOUT_EXPERT) == 0   # E > 1024
    st, h = abi.moe_a2a_create_layout(c, abi.MOE_LAYOUT_EXPERT, 1 << 30, ex)
    assert st == abi.MOE_OK
    assert abi.moe_a2a_set_reduction(h, abi.MOE_REDUCE_BF16_TOPK_TREE) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_set_reduction(h, abi.MOE_REDUCE_FP32_RANK_ORDER) == abi.MOE_OK
    abi.moe_a2a_destroy(h)
    assert abi.moe_a2a_create_layout(c, 5, 1 << 30, ex)[0] == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_a2a_create_layout(c, abi.MOE_LAYOUT_EXPERT, 1 << 30, ex - 1)[0] == \
        abi.MOE_ERR_CAPACITY


def test_expert_gemm_host_checks(abi):
    A = 1 << 20
    assert abi.moe_expert_gemm(None, A, 128, 0) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_expert_gemm_fp8(None, A, A, 128, 0) == abi.MOE_ERR_INVALID_ARG
    c = abi.config(4, 64, 256, 16, 2)
    need = abi.moe_a2a_workspace_bytes_layout(c, abi.MOE_LAYOUT_EXPERT)
    st, h = abi.moe_a2a_create_layout(c, abi.MOE_LAYOUT_EXPERT, 1 << 30, need)
    assert st == abi.MOE_OK
    # no dispatch pending: the phase error comes first, nothing is queued
    assert abi.moe_expert_gemm(h, A, 256, 0) == abi.MOE_ERR_PHASE
    assert abi.moe_expert_gemm_fp8(h, A, A, 256, 0) == abi.MOE_ERR_PHASE
    assert abi.moe_a2a_phase(h) == 0
    abi.moe_a2a_destroy(h)


def _regions_total(sizes):
    off = 0
    for b in sizes:
        off = (off + b + 255) // 256 * 256
    return off


@pytest.mark.parametrize("R,M,H,E,K", [(8, 4096, 7168, 256, 8), (6, 300, 136, 48, 5),
                                       (32, 48, 64, 256, 32)])
def test_workspace_is_the_documented_regions(abi, R, M, H, E, K):
    # The rank layout's regions, each 256-byte aligned, in the order the
    # design notes list them: receive rows, combine payload, metadata rows,
    # scales, source map, counts (two local-expert count buffers: the
    # one-launch dispatch alternates them), send table and weights, top-k slot ranks,
    # per-tile counts and prefixes (tiles of 32 tokens, the smallest routing
    # tile), per-source tickets and expert accumulators, tile-local slots,
    # the flag word.
    RP = (R + 3) // 4 * 4
    NT = (M + 31) // 32
    rank = [R * R * M * H * 2, R * R * M * H * 2, R * R * M * K * 4, R * R * M * K * 4,
            R * R * M * 4, R * R * M * 4, R * R * 4, E * 4, E * 4, R * M * RP * 4,
            R * M * RP * 4, R * M * K, R * NT * RP * 4, R * NT * RP * 4, R * 4, R * E * 4,
            R * M * RP * 4, 256]
    c = abi.config(R, M, H, E, K)
    assert abi.moe_a2a_workspace_bytes(c) == _regions_total(rank)
    # Expert layout: per-expert planes of cap = R * M rows, rows per expert
    # and the expert histogram (two pairs: the one-launch dispatch alternates
    # them), send table of KP entries per token, per-tile expert counts
    # (256-token tiles), the expert histogram accumulator, the flag word.
    if E <= 1024 and E * R * M < 2 ** 31:
        KP = (K + 3) // 4 * 4
        cap, NTe = R * M, (M + 255) // 256
        ex = [E * cap * H * 2, E * cap * H * 2, E * cap * 4, E * cap * 4, E * cap * 4, E * 4,
              E * 4, E * 4, E * 4, R * M * KP * 4, R * M * KP * 4, R * NTe * E * 4, E * 4, 256]
        assert abi.moe_a2a_workspace_bytes_layout(c, abi.MOE_LAYOUT_EXPERT) == \
            _regions_total(ex)


def test_expert_gemm_rank_host_checks(abi):
    # scratch: pair cursors [E] and the count of rows with several local
    # experts, the receive row and gate mark of each pair [R*M*K] each, the
    # pair of each (row, k) [R*R*M*K], the list of rows with several local
    # experts [R*M*(K/2)] (each holds two pairs or more) and the pair-major
    # bf16 outputs [R*M*K][N]
    R, M, H, E, K, N = 8, 64, 256, 32, 4, 384
    c = abi.config(R, M, H, E, K)
    assert abi.moe_expert_gemm_rank_scratch_bytes(c, N) == _regions_total(
        [(E + 1) * 4, R * M * K * 4, R * M * K * 4, R * R * M * K * 4, R * M * (K // 2) * 4,
         R * M * K * N * 2])
    c3 = abi.config(R, M, H, E, 3)  # odd top-k: floor(K / 2) list entries per token
    assert abi.moe_expert_gemm_rank_scratch_bytes(c3, N) == _regions_total(
        [(E + 1) * 4, R * M * 3 * 4, R * M * 3 * 4, R * R * M * 3 * 4, R * M * 1 * 4,
         R * M * 3 * N * 2])
    assert abi.moe_expert_gemm_rank_scratch_bytes(c, 100) == 0        # N % 128
    A = 1 << 20
    assert abi.moe_expert_gemm_rank(None, A, 256, 1, 0, A, 1 << 30) == abi.MOE_ERR_INVALID_ARG
    need = abi.moe_a2a_workspace_bytes(c)
    st, h = abi.moe_a2a_create(c, 1 << 30, need)
    assert st == abi.MOE_OK
    # no dispatch pending: the phase error comes first, nothing is queued
    assert abi.moe_expert_gemm_rank(h, A, 256, 1, 0, A, 1 << 30) == abi.MOE_ERR_PHASE
    assert abi.moe_a2a_phase(h) == 0
    abi.moe_a2a_destroy(h)
    # the expert layout has its own product
    ex = abi.moe_a2a_workspace_bytes_layout(c, abi.MOE_LAYOUT_EXPERT)
    st, h = abi.moe_a2a_create_layout(c, abi.MOE_LAYOUT_EXPERT, 1 << 30, ex)
    assert st == abi.MOE_OK
    assert abi.moe_expert_gemm_rank(h, A, 256, 1, 0, A, 1 << 30) == abi.MOE_ERR_PHASE
    abi.moe_a2a_destroy(h)


def test_owner_multiply_high_is_exact():
    # The kernels find an expert's owner rank e // Epr as (e * ceil(2^32 / Epr)) >> 32
    # (owner_magic in kernels.h).  Exact for e * Epr < 2^32: every expert id and every
    # Epr allowed by MOE_MAX_EXPERTS = 8192, checked exhaustively.
    e = np.arange(8192, dtype=np.uint64)
    for D in range(1, 8193):
        magic = np.uint64(((1 << 32) + D - 1) // D)
        assert np.array_equal((e * magic) >> np.uint64(32), e // np.uint64(D)), D
