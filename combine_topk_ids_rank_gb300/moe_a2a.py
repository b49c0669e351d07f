"""Thin ctypes binding of the C ABI in include/moe_a2a.h (libmoe_a2a.so).

The module-level functions carry the C names and take raw device pointers
(ints) and sizes; they return the C status codes.  `MoeA2A` wraps them for
torch tensors: it allocates the workspace with torch, checks dtypes, shapes
and devices, passes data pointers and the current CUDA stream, and raises
`MoeA2AError` on any status other than MOE_OK.  Every step of the path runs
in the library's CUDA kernels; there is no fallback: if the library is
missing, importing this module fails.
"""
import ctypes
import os

LIBRARY = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_a2a.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_PHASE = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_CUDA = 4
MOE_ERR_ROUTING = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_INTERNAL = 7
MOE_ERR_SETUP_IN_CAPTURE = 8
MOE_DEVICE_FLAG_BAD_EXPERT_ID = 0x1
MOE_DEVICE_FLAG_WAIT_TIMEOUT = 0x2
MOE_DEVICE_FLAG_BAD_SLOT = 0x4

EXPORTS = ("moe_a2a_workspace_bytes", "moe_a2a_create", "moe_dispatch",
           "moe_combine_payload", "moe_combine", "moe_a2a_get_error",
           "moe_a2a_destroy", "moe_a2a_phase", "moe_a2a_status_string",
           "moe_route_static_scratch_bytes", "moe_route_static_scratch",
           "moe_a2a_set_reduction", "moe_dispatch_varlen", "moe_a2a_set_active_ranks",
           "moe_a2a_set_recv_format", "moe_combine_fp8", "moe_quantize_rows_fp8",
           "moe_a2a_workspace_bytes_layout", "moe_a2a_create_layout",
           "moe_expert_gemm", "moe_expert_gemm_fp8", "moe_expert_gemm_rank_scratch_bytes",
           "moe_expert_gemm_rank", "moe_expert_gemm_rank_fp8")
MOE_REDUCE_FP32_RANK_ORDER = 0
MOE_REDUCE_BF16_TOPK_TREE = 1
MOE_STATIC_SCRATCH_BYTES = 4 << 20
MOE_FORMAT_BF16 = 0
MOE_FORMAT_FP8_E4M3 = 1
MOE_LAYOUT_RANK = 0
MOE_LAYOUT_EXPERT = 1


class MoeA2AConfig(ctypes.Structure):
    _fields_ = [("ep_size", ctypes.c_int32), ("max_tokens_per_rank", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]


class MoeDispatchView(ctypes.Structure):
    _fields_ = [("recv_x", ctypes.c_void_p), ("recv_topk_ids", ctypes.c_void_p),
                ("recv_topk_w", ctypes.c_void_p), ("src_token", ctypes.c_void_p),
                ("recv_counts", ctypes.c_void_p), ("local_expert_counts", ctypes.c_void_p),
                ("send_slot", ctypes.c_void_p), ("dest_weight", ctypes.c_void_p),
                ("plane_stride", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int32),
                ("send_stride", ctypes.c_int32), ("token_stride", ctypes.c_int32),
                ("recv_scale", ctypes.c_void_p), ("recv_format", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("kernels", ctypes.c_int32)]


class MoeA2AError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (where, status_string(status), status))


def _load(path: str = LIBRARY):
    if not os.path.exists(path):
        raise ImportError("libmoe_a2a.so is not built (%s); run __graft_entry__.build()" % path)
    # torch first, so that the CUDA runtime it loaded is the one the library binds to
    try:
        import torch  # noqa: F401
    except ImportError:
        pass
    lib = ctypes.CDLL(path)
    p, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    cfgp = ctypes.POINTER(MoeA2AConfig)
    lib.moe_a2a_workspace_bytes.argtypes = [cfgp]
    lib.moe_a2a_workspace_bytes.restype = sz
    lib.moe_a2a_create.argtypes = [cfgp, p, sz, ctypes.POINTER(p)]
    lib.moe_a2a_create.restype = ctypes.c_int
    lib.moe_a2a_workspace_bytes_layout.argtypes = [cfgp, i32]
    lib.moe_a2a_workspace_bytes_layout.restype = sz
    lib.moe_a2a_create_layout.argtypes = [cfgp, i32, p, sz, ctypes.POINTER(p)]
    lib.moe_a2a_create_layout.restype = ctypes.c_int
    lib.moe_dispatch.argtypes = [p, p, p, p, i32, i32, p, ctypes.POINTER(MoeDispatchView)]
    lib.moe_dispatch.restype = ctypes.c_int
    lib.moe_combine_payload.argtypes = [p]
    lib.moe_combine_payload.restype = p
    lib.moe_combine.argtypes = [p, p, i32, p, p, ctypes.c_float, p, p, p]
    lib.moe_combine.restype = ctypes.c_int
    lib.moe_a2a_get_error.argtypes = [p, p, ctypes.POINTER(ctypes.c_uint32)]
    lib.moe_a2a_get_error.restype = ctypes.c_int
    lib.moe_a2a_destroy.argtypes = [p]
    lib.moe_a2a_destroy.restype = ctypes.c_int
    lib.moe_a2a_phase.argtypes = [p]
    lib.moe_a2a_phase.restype = ctypes.c_int
    lib.moe_dispatch_varlen.argtypes = [p, p, p, p, ctypes.POINTER(ctypes.c_int32), i32, p,
                                        ctypes.POINTER(MoeDispatchView)]
    lib.moe_dispatch_varlen.restype = ctypes.c_int
    lib.moe_a2a_set_active_ranks.argtypes = [p, ctypes.c_uint32]
    lib.moe_a2a_set_active_ranks.restype = ctypes.c_int
    lib.moe_combine_fp8.argtypes = [p, p, i32, p, p, ctypes.c_float, p, p, p, p]
    lib.moe_combine_fp8.restype = ctypes.c_int
    lib.moe_quantize_rows_fp8.argtypes = [p, ctypes.c_int64, i32, p, p, p]
    lib.moe_quantize_rows_fp8.restype = ctypes.c_int
    lib.moe_expert_gemm.argtypes = [p, p, i32, p, p]
    lib.moe_expert_gemm.restype = ctypes.c_int
    lib.moe_expert_gemm_fp8.argtypes = [p, p, p, i32, p, p]
    lib.moe_expert_gemm_fp8.restype = ctypes.c_int
    lib.moe_expert_gemm_rank_scratch_bytes.argtypes = [ctypes.POINTER(MoeA2AConfig), i32]
    lib.moe_expert_gemm_rank_scratch_bytes.restype = ctypes.c_size_t
    lib.moe_expert_gemm_rank.argtypes = [p, p, i32, i32, p, p, ctypes.c_size_t, p]
    lib.moe_expert_gemm_rank.restype = ctypes.c_int
    lib.moe_expert_gemm_rank_fp8.argtypes = [p, p, p, i32, i32, p, p, ctypes.c_size_t, p]
    lib.moe_expert_gemm_rank_fp8.restype = ctypes.c_int
    lib.moe_a2a_set_recv_format.argtypes = [p, i32]
    lib.moe_a2a_set_recv_format.restype = ctypes.c_int
    lib.moe_a2a_set_reduction.argtypes = [p, i32]
    lib.moe_a2a_set_reduction.restype = ctypes.c_int
    lib.moe_a2a_status_string.argtypes = [ctypes.c_int]
    lib.moe_a2a_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


# ---- the C ABI, one function per entry point ---------------------------------

def config(ep_size, max_tokens_per_rank, hidden, num_experts, top_k) -> MoeA2AConfig:
    return MoeA2AConfig(ep_size, max_tokens_per_rank, hidden, num_experts, top_k)


def moe_a2a_workspace_bytes(cfg: MoeA2AConfig) -> int:
    return int(_lib.moe_a2a_workspace_bytes(ctypes.byref(cfg)))


def moe_a2a_create(cfg: MoeA2AConfig, d_workspace: int, workspace_bytes: int):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = _lib.moe_a2a_create(ctypes.byref(cfg), ctypes.c_void_p(d_workspace),
                             workspace_bytes, ctypes.byref(h))
    return st, h


def moe_a2a_workspace_bytes_layout(cfg: MoeA2AConfig, layout: int) -> int:
    return int(_lib.moe_a2a_workspace_bytes_layout(ctypes.byref(cfg), layout))


def moe_a2a_create_layout(cfg: MoeA2AConfig, layout: int, d_workspace: int,
                          workspace_bytes: int):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = _lib.moe_a2a_create_layout(ctypes.byref(cfg), layout, ctypes.c_void_p(d_workspace),
                                    workspace_bytes, ctypes.byref(h))
    return st, h


def moe_dispatch(h, d_topk_ids: int, d_topk_w: int, d_x: int, tokens_per_rank: int,
                 runtime_max_tokens_per_rank: int, stream: int = 0):
    """Returns (status, MoeDispatchView)."""
    view = MoeDispatchView()
    st = _lib.moe_dispatch(h, ctypes.c_void_p(d_topk_ids), ctypes.c_void_p(d_topk_w),
                           ctypes.c_void_p(d_x), tokens_per_rank, runtime_max_tokens_per_rank,
                           ctypes.c_void_p(stream), ctypes.byref(view))
    return st, view


def moe_dispatch_varlen(h, d_topk_ids: int, d_topk_w: int, d_x: int, tokens_per_rank,
                        runtime_max_tokens_per_rank: int, stream: int = 0):
    """Returns (status, MoeDispatchView); tokens_per_rank is a host sequence."""
    view = MoeDispatchView()
    counts = (ctypes.c_int32 * len(tokens_per_rank))(*[int(c) for c in tokens_per_rank])
    st = _lib.moe_dispatch_varlen(h, ctypes.c_void_p(d_topk_ids), ctypes.c_void_p(d_topk_w),
                                  ctypes.c_void_p(d_x), counts, runtime_max_tokens_per_rank,
                                  ctypes.c_void_p(stream), ctypes.byref(view))
    return st, view


def moe_a2a_set_active_ranks(h, active: int) -> int:
    return _lib.moe_a2a_set_active_ranks(h, active)


def moe_combine_payload(h) -> int:
    return _lib.moe_combine_payload(h) or 0


def moe_combine(h, d_expert_out: int, weighted: bool, d_residual: int, d_gamma: int, eps: float,
                d_out: int, d_residual_out: int, stream: int = 0) -> int:
    return _lib.moe_combine(h, ctypes.c_void_p(d_expert_out), int(bool(weighted)),
                            ctypes.c_void_p(d_residual), ctypes.c_void_p(d_gamma),
                            float(eps), ctypes.c_void_p(d_out), ctypes.c_void_p(d_residual_out),
                            ctypes.c_void_p(stream))


def moe_combine_fp8(h, d_expert_out: int, weighted: bool, d_residual: int, d_gamma: int,
                    eps: float, d_out_fp8: int, d_out_scale: int, d_residual_out: int,
                    stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_combine_fp8(h, v(d_expert_out), int(bool(weighted)), v(d_residual),
                                v(d_gamma), float(eps), v(d_out_fp8), v(d_out_scale),
                                v(d_residual_out), v(stream))


def moe_quantize_rows_fp8(d_x: int, rows: int, hidden: int, d_q: int, d_scale: int,
                          stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_quantize_rows_fp8(v(d_x), rows, hidden, v(d_q), v(d_scale), v(stream))


def quantize_rows_fp8(x, out=None, scale=None, stream=None):
    """fp32 [..., H] CUDA tensor -> (float8_e4m3fn [..., H], float32 [...])."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    H = x.shape[-1]
    rows = x.numel() // H if H else 0
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    st = moe_quantize_rows_fp8(x.data_ptr(), rows, H, out.data_ptr(), scale.data_ptr(),
                               stream.cuda_stream if hasattr(stream, "cuda_stream")
                               else int(stream))
    if st != MOE_OK:
        raise MoeA2AError(st, "moe_quantize_rows_fp8")
    return out, scale


def moe_expert_gemm(h, d_w: int, N: int, d_out: int, stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_expert_gemm(h, v(d_w), N, v(d_out), v(stream))


def moe_expert_gemm_rank_scratch_bytes(cfg: MoeA2AConfig, N: int) -> int:
    return _lib.moe_expert_gemm_rank_scratch_bytes(ctypes.byref(cfg), N)


def moe_expert_gemm_rank(h, d_w: int, N: int, apply_gates: int, d_out: int, d_scratch: int,
                         scratch_bytes: int, stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_expert_gemm_rank(h, v(d_w), N, apply_gates, v(d_out), v(d_scratch),
                                     scratch_bytes, v(stream))


def moe_expert_gemm_rank_fp8(h, d_w8: int, d_w_scale: int, N: int, apply_gates: int,
                             d_out: int, d_scratch: int, scratch_bytes: int,
                             stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_expert_gemm_rank_fp8(h, v(d_w8), v(d_w_scale), N, apply_gates, v(d_out),
                                         v(d_scratch), scratch_bytes, v(stream))


def moe_expert_gemm_fp8(h, d_w8: int, d_w_scale: int, N: int, d_out: int,
                        stream: int = 0) -> int:
    v = ctypes.c_void_p
    return _lib.moe_expert_gemm_fp8(h, v(d_w8), v(d_w_scale), N, v(d_out), v(stream))


def moe_a2a_set_recv_format(h, fmt: int) -> int:
    return _lib.moe_a2a_set_recv_format(h, fmt)


def moe_a2a_get_error(h, stream: int = 0):
    """Returns (status, device flag bits)."""
    flags = ctypes.c_uint32(0)
    st = _lib.moe_a2a_get_error(h, ctypes.c_void_p(stream), ctypes.byref(flags))
    return st, int(flags.value)


def moe_a2a_destroy(h) -> int:
    return _lib.moe_a2a_destroy(h)


def moe_a2a_phase(h) -> int:
    return _lib.moe_a2a_phase(h)


def moe_a2a_set_reduction(h, reduction: int) -> int:
    return _lib.moe_a2a_set_reduction(h, reduction)


def status_string(status: int) -> str:
    return _lib.moe_a2a_status_string(status).decode()


def moe_route_static_scratch_bytes(ep_size: int, num_experts: int, tokens_per_rank: int) -> int:
    f = _lib.moe_route_static_scratch_bytes
    f.argtypes = [ctypes.c_int32] * 3
    f.restype = ctypes.c_size_t
    return int(f(ep_size, num_experts, tokens_per_rank))


def moe_route_static_scratch(ep_size: int, num_experts: int, top_k: int, tokens_per_rank: int,
                             runtime_max_tokens_per_rank: int, d_topk_ids: int, d_topk_w: int,
                             d_send_slot: int, d_dest_weight: int, d_src_token: int,
                             d_recv_counts: int, d_local_expert_counts: int,
                             d_recv_topk_ids: int, d_recv_topk_w: int, d_flags: int = 0,
                             stream: int = 0) -> int:
    """The routing pass with no device allocation (see include/moe_a2a.h):
    every buffer is the caller's, the temporary memory is the library's
    fixed device array.  Returns the C status code."""
    f = _lib.moe_route_static_scratch
    f.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_void_p] * 11
    f.restype = ctypes.c_int
    v = ctypes.c_void_p
    return f(ep_size, num_experts, top_k, tokens_per_rank, runtime_max_tokens_per_rank,
             v(d_topk_ids), v(d_topk_w), v(d_send_slot), v(d_dest_weight), v(d_src_token),
             v(d_recv_counts), v(d_local_expert_counts), v(d_recv_topk_ids), v(d_recv_topk_w),
             v(d_flags), v(stream))


# ---- torch convenience wrapper ------------------------------------------------

def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


class DispatchView:
    """torch views into the workspace produced by one dispatch."""

    def __init__(self, owner, raw: MoeDispatchView):
        import torch
        R, K, E = owner.ep_size, owner.top_k, owner.num_experts
        H, m, RP = owner.hidden, raw.plane_stride, raw.send_stride
        T = raw.token_stride

        def region(ptr, dtype, shape):
            n = 1
            for s in shape:
                n *= s
            off = ptr - owner.workspace.data_ptr()
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            return owner.workspace[off:off + nbytes].view(dtype).view(shape)

        self.plane_stride, self.send_stride = m, RP
        self.tokens_per_rank, self.token_stride = raw.tokens_per_rank, T
        self.recv_format, self.layout = raw.recv_format, raw.layout
        self.kernels = raw.kernels
        # planes: (dst rank, src rank) of m rows, or (expert) of cap = m rows
        planes = (E,) if raw.layout == MOE_LAYOUT_EXPERT else (R, R)
        if raw.recv_format == MOE_FORMAT_FP8_E4M3:
            self.recv_x = region(raw.recv_x, torch.float8_e4m3fn, planes + (m, H))
            self.recv_scale = region(raw.recv_scale, torch.float32, planes + (m,))
        else:
            self.recv_x = region(raw.recv_x, torch.bfloat16, planes + (m, H))
            self.recv_scale = None
        if raw.layout == MOE_LAYOUT_EXPERT:
            self.recv_topk_ids = None
            self.recv_topk_w = region(raw.recv_topk_w, torch.float32, (E, m))
            self.src_token = region(raw.src_token, torch.int32, (E, m))
            self.recv_counts = region(raw.recv_counts, torch.int32, (E,))
            self.local_expert_counts = region(raw.local_expert_counts, torch.int32, (E,))
        else:
            self.recv_topk_ids = region(raw.recv_topk_ids, torch.int32, (R, R, m, K))
            self.recv_topk_w = region(raw.recv_topk_w, torch.float32, (R, R, m, K))
            self.src_token = region(raw.src_token, torch.int32, (R, R, m))
            self.recv_counts = region(raw.recv_counts, torch.int32, (R, R))
            self.local_expert_counts = region(raw.local_expert_counts, torch.int32,
                                              (R, E // R))
        self.send_slot = region(raw.send_slot, torch.int32, (R, T, RP))
        self.dest_weight = region(raw.dest_weight, torch.float32, (R, T, RP))


class MoeA2A:
    """One dispatch/combine handle over a torch-allocated device workspace."""

    def __init__(self, ep_size: int, max_tokens_per_rank: int, hidden: int, num_experts: int,
                 top_k: int, device=None, layout: int = MOE_LAYOUT_RANK):
        import torch
        self.ep_size, self.max_tokens_per_rank, self.hidden = ep_size, max_tokens_per_rank, hidden
        self.num_experts, self.top_k, self.layout = num_experts, top_k, layout
        self.cfg = config(ep_size, max_tokens_per_rank, hidden, num_experts, top_k)
        nbytes = moe_a2a_workspace_bytes_layout(self.cfg, layout)
        if nbytes == 0:
            raise MoeA2AError(MOE_ERR_INVALID_ARG, "moe_a2a_workspace_bytes_layout")
        self.device = torch.device(device if device is not None else "cuda")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        st, self.handle = moe_a2a_create_layout(self.cfg, layout, self.workspace.data_ptr(),
                                                nbytes)
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_a2a_create")
        self.last_view = None
        self._views = {}
        self._payload = None

    def _stream(self, stream) -> int:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

    def _check(self, t, dtype, shape, name):
        if t.dtype != dtype or tuple(t.shape) != tuple(shape):
            raise ValueError("%s: expected %s %s, got %s %s" % (name, dtype, tuple(shape),
                                                               t.dtype, tuple(t.shape)))
        if not t.is_contiguous() or t.device != self.workspace.device:
            raise ValueError("%s must be contiguous on %s" % (name, self.workspace.device))

    def _planes(self):
        return (self.num_experts,) if self.layout == MOE_LAYOUT_EXPERT else (
            self.ep_size, self.ep_size)

    @property
    def phase(self) -> int:
        return moe_a2a_phase(self.handle)

    def dispatch(self, topk_ids, topk_w, x, runtime_max_tokens_per_rank: int = None,
                 stream=None) -> DispatchView:
        import torch
        R, H, K = self.ep_size, self.hidden, self.top_k
        T = topk_ids.shape[1]
        m = T if runtime_max_tokens_per_rank is None else runtime_max_tokens_per_rank
        self._check(topk_ids, torch.int32, (R, T, K), "topk_ids")
        self._check(topk_w, torch.float32, (R, T, K), "topk_w")
        self._check(x, torch.bfloat16, (R, T, H), "x")
        st, raw = moe_dispatch(self.handle, _ptr(topk_ids), _ptr(topk_w), _ptr(x), T, m,
                               self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_dispatch")
        return self._view(raw)

    def _view(self, raw) -> DispatchView:
        # The views depend only on (m, token stride, format) and on which of
        # the two count regions holds this call's local-expert counts: reuse
        # them across calls.
        key = (raw.plane_stride, raw.token_stride, raw.recv_format, raw.local_expert_counts)
        view = self._views.get(key)
        if view is None:
            view = self._views[key] = DispatchView(self, raw)
        else:  # the per-call scalars of this call
            view.kernels, view.tokens_per_rank = raw.kernels, raw.tokens_per_rank
        self.last_view = view
        return view

    def dispatch_varlen(self, topk_ids, topk_w, x, tokens_per_rank, stream=None) -> DispatchView:
        """Per-rank token counts: inputs [R, m, ...], rows t < tokens_per_rank[s]."""
        import torch
        R, H, K = self.ep_size, self.hidden, self.top_k
        m = topk_ids.shape[1]
        self._check(topk_ids, torch.int32, (R, m, K), "topk_ids")
        self._check(topk_w, torch.float32, (R, m, K), "topk_w")
        self._check(x, torch.bfloat16, (R, m, H), "x")
        st, raw = moe_dispatch_varlen(self.handle, _ptr(topk_ids), _ptr(topk_w), _ptr(x),
                                      list(tokens_per_rank), m, self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_dispatch_varlen")
        return self._view(raw)

    def set_active_ranks(self, active: int):
        """Bit d set = logical rank d alive (default: all)."""
        st = moe_a2a_set_active_ranks(self.handle, active)
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_a2a_set_active_ranks")

    def combine_payload(self):
        """bf16 [R, R, m, H] view of the in-workspace combine payload region."""
        import torch
        if self.last_view is None:
            raise RuntimeError("no dispatch yet")
        R, H, m = self.ep_size, self.hidden, self.last_view.plane_stride
        planes = (self.num_experts,) if self.layout == MOE_LAYOUT_EXPERT else (R, R)
        if self._payload is None or self._payload.shape[-2] != m:
            off = moe_combine_payload(self.handle) - self.workspace.data_ptr()
            n = planes[0] * (planes[1] if len(planes) > 1 else 1) * m * H * 2
            self._payload = self.workspace[off:off + n].view(torch.bfloat16).view(
                *planes, m, H)
        return self._payload

    def combine(self, expert_out=None, weighted: bool = False, residual=None, gamma=None,
                eps: float = 1e-6, out=None, residual_out=None, stream=None):
        import torch
        if self.last_view is None:
            st = moe_combine(self.handle, 0, weighted, 0, 0, eps, 0, 0, self._stream(stream))
            raise MoeA2AError(st if st != MOE_OK else MOE_ERR_PHASE, "moe_combine")
        R, H = self.ep_size, self.hidden
        T, m = self.last_view.token_stride, self.last_view.plane_stride
        if expert_out is not None:
            self._check(expert_out, torch.bfloat16, self._planes() + (m, H), "expert_out")
        if residual is not None:
            self._check(residual, torch.bfloat16, (R, T, H), "residual")
            self._check(gamma, torch.bfloat16, (H,), "gamma")
            if residual_out is not None:
                self._check(residual_out, torch.bfloat16, (R, T, H), "residual_out")
        if out is None:
            out = torch.empty((R, T, H), dtype=torch.bfloat16, device=self.workspace.device)
        self._check(out, torch.bfloat16, (R, T, H), "out")
        st = moe_combine(self.handle, _ptr(expert_out), weighted, _ptr(residual), _ptr(gamma),
                         eps, _ptr(out), _ptr(residual_out), self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_combine")
        return out

    def combine_fp8(self, expert_out=None, weighted: bool = False, residual=None, gamma=None,
                    eps: float = 1e-6, out=None, out_scale=None, residual_out=None,
                    stream=None):
        """As combine, with an e4m3 output and one fp32 scale per token row:
        returns (out float8_e4m3fn [R, T, H], out_scale float32 [R, T])."""
        import torch
        if self.last_view is None:
            st = moe_combine_fp8(self.handle, 0, weighted, 0, 0, eps, 0, 0, 0,
                                 self._stream(stream))
            raise MoeA2AError(st if st != MOE_OK else MOE_ERR_PHASE, "moe_combine_fp8")
        R, H = self.ep_size, self.hidden
        T, m = self.last_view.token_stride, self.last_view.plane_stride
        if expert_out is not None:
            self._check(expert_out, torch.bfloat16, self._planes() + (m, H), "expert_out")
        if residual is not None:
            self._check(residual, torch.bfloat16, (R, T, H), "residual")
            self._check(gamma, torch.bfloat16, (H,), "gamma")
            if residual_out is not None:
                self._check(residual_out, torch.bfloat16, (R, T, H), "residual_out")
        dev = self.workspace.device
        if out is None:
            out = torch.empty((R, T, H), dtype=torch.float8_e4m3fn, device=dev)
        if out_scale is None:
            out_scale = torch.empty((R, T), dtype=torch.float32, device=dev)
        self._check(out, torch.float8_e4m3fn, (R, T, H), "out")
        self._check(out_scale, torch.float32, (R, T), "out_scale")
        st = moe_combine_fp8(self.handle, _ptr(expert_out), weighted, _ptr(residual),
                             _ptr(gamma), eps, _ptr(out), _ptr(out_scale), _ptr(residual_out),
                             self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_combine_fp8")
        return out, out_scale

    def expert_gemm(self, w, out=None, stream=None):
        """Expert layout: out[e][j] = x[e][j] . w[e]^T for the received rows.
        w: bf16 [E, N, H]; out: bf16 [E, cap, N], or None to write the
        combine payload (N == H).  Returns the output tensor."""
        import torch
        E, H = self.num_experts, self.hidden
        N = w.shape[1]
        self._check(w, torch.bfloat16, (E, N, H), "w")
        if out is not None:
            self._check(out, torch.bfloat16, (E, self.last_view.plane_stride, N), "out")
        st = moe_expert_gemm(self.handle, _ptr(w), N, _ptr(out), self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_expert_gemm")
        return out if out is not None else self.combine_payload()

    def _rank_out_scratch(self, N, out, scratch):
        import torch
        R = self.ep_size
        if out is not None:
            self._check(out, torch.bfloat16, (R, R, self.last_view.plane_stride, N), "out")
        need = moe_expert_gemm_rank_scratch_bytes(self.cfg, N)
        if need == 0:
            raise MoeA2AError(MOE_ERR_INVALID_ARG, "moe_expert_gemm_rank_scratch_bytes")
        if scratch is None:
            if getattr(self, "_rank_scratch", None) is None or self._rank_scratch.numel() < need:
                self._rank_scratch = torch.empty(need, dtype=torch.uint8, device=self.device)
            scratch = self._rank_scratch
        if scratch.dtype != torch.uint8 or scratch.device != self.workspace.device:
            raise ValueError("scratch: expected a uint8 tensor on %s" % self.workspace.device)
        return scratch

    def expert_gemm_rank(self, w, apply_gates=True, out=None, scratch=None, stream=None):
        """Rank layout: each received row's local experts applied to it, their
        bf16 outputs summed with the gates (or plainly) in ascending top-k
        order.  w: bf16 [E, N, H]; out: bf16 [R, R, m, N], or None to write the
        combine payload (N == H); scratch: uint8 device tensor of at least
        moe_expert_gemm_rank_scratch_bytes bytes (allocated and kept here if
        None).  Returns the output tensor."""
        import torch
        E, H = self.num_experts, self.hidden
        N = w.shape[1]
        self._check(w, torch.bfloat16, (E, N, H), "w")
        scratch = self._rank_out_scratch(N, out, scratch)
        st = moe_expert_gemm_rank(self.handle, _ptr(w), N, int(bool(apply_gates)), _ptr(out),
                                  scratch.data_ptr(), scratch.numel(), self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_expert_gemm_rank")
        return out if out is not None else self.combine_payload()

    def expert_gemm_rank_fp8(self, w8, w_scale, apply_gates=True, out=None, scratch=None,
                             stream=None):
        """expert_gemm_rank on FP8 operands, for a rank-layout dispatch in the
        FP8 receive format: each expert output is (qx . qw[e]^T) sx sw[e],
        narrowed to bf16, then gated and summed as expert_gemm_rank does.
        w8: e4m3 [E, N, H] (float8_e4m3fn or uint8); w_scale: float32 [E, N];
        out and scratch as for expert_gemm_rank."""
        import torch
        E, H = self.num_experts, self.hidden
        N = w8.shape[1]
        if w8.dtype not in (torch.float8_e4m3fn, torch.uint8) or tuple(w8.shape) != (E, N, H) \
                or not w8.is_contiguous():
            raise ValueError("w8: expected contiguous e4m3 [%d, N, %d]" % (E, H))
        self._check(w_scale, torch.float32, (E, N), "w_scale")
        scratch = self._rank_out_scratch(N, out, scratch)
        st = moe_expert_gemm_rank_fp8(self.handle, _ptr(w8), _ptr(w_scale), N,
                                      int(bool(apply_gates)), _ptr(out), scratch.data_ptr(),
                                      scratch.numel(), self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_expert_gemm_rank_fp8")
        return out if out is not None else self.combine_payload()

    def expert_gemm_fp8(self, w8, w_scale, out=None, stream=None):
        """FP8 receive format: out[e][j] = (qx[e][j] . qw[e]^T) sx[e][j] sw[e].
        w8: e4m3 [E, N, H] (float8_e4m3fn or uint8); w_scale: float32 [E, N];
        out: bf16 [E, cap, N], or None to write the combine payload (N == H)."""
        import torch
        E, H = self.num_experts, self.hidden
        N = w8.shape[1]
        if w8.dtype not in (torch.float8_e4m3fn, torch.uint8) or tuple(w8.shape) != (E, N, H) \
                or not w8.is_contiguous():
            raise ValueError("w8: expected contiguous e4m3 [%d, N, %d]" % (E, H))
        self._check(w_scale, torch.float32, (E, N), "w_scale")
        if out is not None:
            self._check(out, torch.bfloat16, (E, self.last_view.plane_stride, N), "out")
        st = moe_expert_gemm_fp8(self.handle, _ptr(w8), _ptr(w_scale), N, _ptr(out),
                                 self._stream(stream))
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_expert_gemm_fp8")
        return out if out is not None else self.combine_payload()

    def set_recv_format(self, fmt: int):
        """MOE_FORMAT_BF16 (default) or MOE_FORMAT_FP8_E4M3 rows in recv_x."""
        st = moe_a2a_set_recv_format(self.handle, fmt)
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_a2a_set_recv_format")

    def set_reduction(self, reduction: int):
        """MOE_REDUCE_FP32_RANK_ORDER (default) or MOE_REDUCE_BF16_TOPK_TREE."""
        st = moe_a2a_set_reduction(self.handle, reduction)
        if st != MOE_OK:
            raise MoeA2AError(st, "moe_a2a_set_reduction")

    def get_error(self, stream=None):
        """Synchronise, read and clear the device flag word: (status, bits)."""
        return moe_a2a_get_error(self.handle, self._stream(stream))

    def close(self):
        if getattr(self, "handle", None):
            moe_a2a_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
