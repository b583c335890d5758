"""Sparse Mixture-of-Experts layer forward on one B300 (sm_103a).

A thin ctypes binding of ``libmoe.so`` (C ABI in ``include/moe.h``). Every
function here only marshals arguments: tensors become device pointers, the
current torch stream becomes the CUDA stream, and a non-OK status raises
``MoeError``. All computation happens in the library's CUDA kernels; there is
no Python or CPU fallback — importing fails when the library is missing.

torch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import pathlib

import torch  # loads the CUDA runtime that libmoe.so then shares

_LIB_PATH = pathlib.Path(__file__).resolve().with_name("libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_FAULT = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_SOFTMAX_THEN_TOPK, MOE_TOPK_THEN_SOFTMAX = 0, 1
MOE_ACT_SILU_GATED, MOE_ACT_RELU = 0, 1
MOE_ROUTING_TOKEN_CHOICE, MOE_ROUTING_EXPERT_CHOICE = 0, 1
MOE_DEBUG_FORCE_SIMT_FFN = 1
MOE_DEBUG_FFN_PAIR = 2
MOE_DEBUG_FFN_SINGLE = 4
MOE_DEBUG_FFN_SWAP = 8
MOE_DEBUG_NO_PDL = 16
MOE_DEBUG_ROUTER_STALL = 32

EXPORTED = ("moe_validate_config", "moe_workspace_size", "moe_max_rows", "moe_capacity",
            "moe_router_topk", "moe_dispatch", "moe_grouped_ffn", "moe_combine", "moe_forward",
            "moe_forward_profiled", "moe_check_error", "moe_status_str", "moe_router_topk_noalloc",
            "moe_router_topk_train", "moe_router_shard_stats", "moe_router_shard_assign",
            "moe_router_expert_choice", "moe_combine_expert_choice", "moe_backward",
            "moe_backward_workspace_size", "moe_forward_graph_create", "moe_forward_graph_launch",
            "moe_forward_graph_destroy", "moe_router_workspace_size",
            "moe_router_noalloc_check_error", "moe_preact_offset")


class moe_config(ctypes.Structure):
    """Mirror of the C struct moe_config (all fields int32)."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "d", "N", "k", "h", "h_shared", "dtype", "gating", "act", "cap_num", "cap_den",
        "has_router_bias", "debug_flags", "routing", "save_preact")]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


def _load() -> ctypes.CDLL:
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH.name} is not built; run "
                          "`python -m sparse_mixture_experts_64_b300.build`")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P, I32, SZ, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int64
    cfgp = ctypes.POINTER(moe_config)
    sig = {
        "moe_validate_config": (I32, [cfgp]),
        "moe_workspace_size": (SZ, [cfgp]),
        "moe_router_workspace_size": (SZ, [cfgp]),
        "moe_preact_offset": (SZ, [cfgp, I32]),
        "moe_router_noalloc_check_error": (I32, [P]),
        "moe_max_rows": (I64, [cfgp]),
        "moe_capacity": (I32, [cfgp]),
        "moe_router_topk": (I32, [cfgp] + [P] * 11 + [P, SZ, P]),
        "moe_router_topk_noalloc": (I32, [cfgp] + [P] * 11 + [P]),
        "moe_router_topk_train": (I32, [cfgp, P, P, P, P, ctypes.c_float] + [P] * 9 + [P, SZ, P]),
        "moe_router_shard_stats": (I32, [cfgp] + [P] * 7 + [P, SZ, P]),
        "moe_router_expert_choice": (I32, [cfgp] + [P] * 8 + [P, SZ, P]),
        "moe_backward_workspace_size": (SZ, [cfgp]),
        "moe_backward": (I32, [cfgp] + [P] * 12 + [ctypes.c_float, ctypes.c_float] + [P] * 9
                         + [P, SZ, P, SZ, P]),
        "moe_combine_expert_choice": (I32, [cfgp] + [P] * 9 + [P, SZ, P]),
        "moe_router_shard_assign": (I32, [cfgp, P, P, I32, P, P, I64] + [P] * 5 + [P, SZ, P]),
        "moe_dispatch": (I32, [cfgp, P, P, P, P, P, SZ, P]),
        "moe_grouped_ffn": (I32, [cfgp, P, P, P, P, P, P, P, SZ, P]),
        "moe_combine": (I32, [cfgp, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_forward": (I32, [cfgp] + [P] * 15 + [P, SZ, P]),
        "moe_forward_profiled": (I32, [cfgp] + [P] * 15 + [P, SZ, P, P, I32]),
        "moe_forward_graph_create": (I32, [cfgp] + [P] * 15 + [P, SZ, P, I32, ctypes.POINTER(P)]),
        "moe_forward_graph_launch": (I32, [P, P]),
        "moe_forward_graph_destroy": (I32, [P]),
        "moe_check_error": (I32, [P, P]),
        "moe_status_str": (ctypes.c_char_p, [I32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


def status_str(s: int) -> str:
    return _lib.moe_status_str(int(s)).decode()


moe_status_str = status_str


def make_config(T, d, N, k, h, h_shared=0, dtype="bf16", gating="topk_then_softmax",
                act="silu_gated", capacity_factor=None, router_bias=False, debug_flags=0,
                routing="token_choice", save_preact=False, **_ignored) -> moe_config:
    """Build a moe_config from plain fields (the names used by the workload table)."""
    c = moe_config()
    c.T, c.d, c.N, c.k, c.h, c.h_shared = T, d, N, k, h, h_shared
    c.dtype = {"f32": MOE_F32, "bf16": MOE_BF16}[dtype] if isinstance(dtype, str) else int(dtype)
    c.gating = ({"softmax_then_topk": MOE_SOFTMAX_THEN_TOPK,
                 "topk_then_softmax": MOE_TOPK_THEN_SOFTMAX}[gating]
                if isinstance(gating, str) else int(gating))
    c.act = ({"silu_gated": MOE_ACT_SILU_GATED, "relu": MOE_ACT_RELU}[act]
             if isinstance(act, str) else int(act))
    c.cap_num, c.cap_den = capacity_factor if capacity_factor else (0, 0)
    c.has_router_bias = 1 if router_bias else 0
    c.debug_flags = debug_flags
    c.routing = ({"token_choice": MOE_ROUTING_TOKEN_CHOICE, "expert_choice": MOE_ROUTING_EXPERT_CHOICE}[routing]
                 if isinstance(routing, str) else int(routing))
    c.save_preact = 1 if save_preact else 0
    return c


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def moe_validate_config(cfg) -> int:
    return _lib.moe_validate_config(ctypes.byref(cfg))


def moe_workspace_size(cfg) -> int:
    return _lib.moe_workspace_size(ctypes.byref(cfg))


def moe_router_workspace_size(cfg) -> int:
    return _lib.moe_router_workspace_size(ctypes.byref(cfg))


def moe_max_rows(cfg) -> int:
    return _lib.moe_max_rows(ctypes.byref(cfg))


def moe_preact_offset(cfg, shared=False) -> int:
    return _lib.moe_preact_offset(ctypes.byref(cfg), 1 if shared else 0)


def preact_view(cfg, ws, shared=False) -> torch.Tensor:
    """The pre-activations moe_forward kept in `ws` (save_preact) as a bf16 tensor view:
    [R_max][W] (routed, dispatch order) or [T][2 h_shared] (shared expert)."""
    off = moe_preact_offset(cfg, shared)
    if off == ctypes.c_size_t(-1).value:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_preact_offset")
    rows = cfg.T if shared else moe_max_rows(cfg)
    width = 2 * cfg.h_shared if shared else (2 * cfg.h if cfg.act == MOE_ACT_SILU_GATED else cfg.h)
    return ws[off:off + rows * width * 2].view(torch.bfloat16).view(rows, width)


def moe_capacity(cfg) -> int:
    return _lib.moe_capacity(ctypes.byref(cfg))


def workspace(cfg, device="cuda") -> torch.Tensor:
    """A zeroed workspace of moe_workspace_size(cfg) bytes (the error word starts at 0)."""
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoeError(moe_validate_config(cfg), "moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_router_topk(cfg, x, w_r, b_r, topk_idx, topk_gate, counts_routed, counts_kept,
                    expert_offsets, slot_row, perm_token, aux, ws, stream=None):
    _check(_lib.moe_router_topk(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(topk_idx),
                                _p(topk_gate), _p(counts_routed), _p(counts_kept),
                                _p(expert_offsets), _p(slot_row), _p(perm_token), _p(aux),
                                _p(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_router_topk")


def moe_router_topk_train(cfg, x, w_r, b_r, noise, noise_weight, topk_idx, topk_gate,
                          counts_routed, counts_kept, expert_offsets, slot_row, perm_token, aux,
                          z_loss, ws, stream=None):
    """moe_router_topk with noisy top-k gating (noise: fp32 [T][N] standard-normal
    draws or None, scaled by noise_weight) and the router z-loss (z_loss: fp32 [1] or
    None)."""
    _check(_lib.moe_router_topk_train(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(noise),
                                      float(noise_weight), _p(topk_idx), _p(topk_gate),
                                      _p(counts_routed), _p(counts_kept), _p(expert_offsets),
                                      _p(slot_row), _p(perm_token), _p(aux), _p(z_loss), _p(ws),
                                      ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_router_topk_train")


def moe_router_shard_stats(cfg, x, w_r, b_r, topk_idx, topk_gate, slot_counts, prob_sums, ws,
                           stream=None):
    """Token-sharded router, phase 1 (see sharded.py): this rank's routing and its
    per-(expert, slot) selection counts [N][k] and softmax sums [N]."""
    _check(_lib.moe_router_shard_stats(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(topk_idx),
                                       _p(topk_gate), _p(slot_counts), _p(prob_sums), _p(ws),
                                       ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_router_shard_stats")


def moe_router_shard_assign(cfg, topk_idx, slot_base, capacity, global_routed, global_prob_sums,
                            global_T, counts_kept, expert_offsets, slot_row, perm_token, aux, ws,
                            stream=None):
    """Token-sharded router, phase 2: capacity decisions at the global priorities
    slot_base [N][k], dispatch order of this rank's selections, global aux."""
    _check(_lib.moe_router_shard_assign(ctypes.byref(cfg), _p(topk_idx), _p(slot_base),
                                        int(capacity), _p(global_routed), _p(global_prob_sums),
                                        int(global_T), _p(counts_kept), _p(expert_offsets),
                                        _p(slot_row), _p(perm_token), _p(aux), _p(ws),
                                        ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_router_shard_assign")


def moe_router_expert_choice(cfg, x, w_r, b_r, expert_offsets, perm_token, row_gate, token_ptr,
                             token_rows, ws, stream=None):
    """Expert Choice router: every expert keeps its min(C, T) highest-scoring tokens."""
    _check(_lib.moe_router_expert_choice(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r),
                                         _p(expert_offsets), _p(perm_token), _p(row_gate),
                                         _p(token_ptr), _p(token_rows), _p(ws),
                                         ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_router_expert_choice")


def moe_combine_expert_choice(cfg, x, y_perm, token_ptr, token_rows, row_gate, shared_w_gate,
                              shared_w_up, shared_w_down, y, ws, stream=None):
    _check(_lib.moe_combine_expert_choice(ctypes.byref(cfg), _p(x), _p(y_perm), _p(token_ptr),
                                          _p(token_rows), _p(row_gate), _p(shared_w_gate),
                                          _p(shared_w_up), _p(shared_w_down), _p(y), _p(ws),
                                          ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_combine_expert_choice")


def backward_workspace(cfg, device="cuda"):
    """Scratch for moe_backward (uint8, 256-byte aligned by the allocator)."""
    import torch
    return torch.empty(int(_lib.moe_backward_workspace_size(ctypes.byref(cfg))), dtype=torch.uint8, device=device)


def moe_backward(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up,
                 shared_w_down, topk_idx, topk_gate, dy, aux_coef, z_coef, dx, dw_r, db_r,
                 dw_gate_or_w1, dw_up, dw_down, dshared_w_gate, dshared_w_up, dshared_w_down, ws,
                 bws, stream=None):
    """Gradients of sum(dy * y) + aux_coef * aux[0] + z_coef * z after moe_forward with the
    same inputs and workspace ws; bws from backward_workspace(cfg)."""
    _check(_lib.moe_backward(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(w_gate_or_w1), _p(w_up),
                             _p(w_down), _p(shared_w_gate), _p(shared_w_up), _p(shared_w_down),
                             _p(topk_idx), _p(topk_gate), _p(dy), float(aux_coef), float(z_coef),
                             _p(dx), _p(dw_r), _p(db_r), _p(dw_gate_or_w1), _p(dw_up), _p(dw_down),
                             _p(dshared_w_gate), _p(dshared_w_up), _p(dshared_w_down), _p(ws),
                             ws.numel() if ws is not None else 0, _p(bws),
                             bws.numel() if bws is not None else 0, _stream(stream)), "moe_backward")


def moe_router_topk_noalloc(cfg, x, w_r, b_r, topk_idx, topk_gate, counts_routed, counts_kept,
                            expert_offsets, slot_row, perm_token, aux, stream=None):
    """moe_router_topk without a workspace, for callers that cannot allocate device
    memory: the router scratch is a static array inside libmoe.so (32 MiB limit)."""
    _check(_lib.moe_router_topk_noalloc(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(topk_idx),
                                        _p(topk_gate), _p(counts_routed), _p(counts_kept),
                                        _p(expert_offsets), _p(slot_row), _p(perm_token), _p(aux),
                                        _stream(stream)), "moe_router_topk_noalloc")


def moe_router_noalloc_check_error(stream=None) -> int:
    """Synchronise the stream, read and clear the error word of the no-allocation router
    on the current device (the status, not raised)."""
    return _lib.moe_router_noalloc_check_error(_stream(stream))


def moe_dispatch(cfg, x, perm_token, expert_offsets, x_perm, ws=None, stream=None):
    _check(_lib.moe_dispatch(ctypes.byref(cfg), _p(x), _p(perm_token), _p(expert_offsets),
                             _p(x_perm), _p(ws), ws.numel() if ws is not None else 0,
                             _stream(stream)), "moe_dispatch")


def moe_grouped_ffn(cfg, x_perm, expert_offsets, w_gate_or_w1, w_up, w_down, y_perm, ws,
                    stream=None):
    _check(_lib.moe_grouped_ffn(ctypes.byref(cfg), _p(x_perm), _p(expert_offsets),
                                _p(w_gate_or_w1), _p(w_up), _p(w_down), _p(y_perm), _p(ws),
                                ws.numel() if ws is not None else 0, _stream(stream)),
           "moe_grouped_ffn")


def moe_combine(cfg, x, y_perm, slot_row, topk_gate, shared_w_gate, shared_w_up, shared_w_down,
                y, ws, stream=None):
    _check(_lib.moe_combine(ctypes.byref(cfg), _p(x), _p(y_perm), _p(slot_row), _p(topk_gate),
                            _p(shared_w_gate), _p(shared_w_up), _p(shared_w_down), _p(y), _p(ws),
                            ws.numel() if ws is not None else 0, _stream(stream)), "moe_combine")


def moe_forward(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up,
                shared_w_down, y, topk_idx, topk_gate, counts_routed, counts_kept, aux, ws,
                stream=None):
    _check(_lib.moe_forward(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r), _p(w_gate_or_w1),
                            _p(w_up), _p(w_down), _p(shared_w_gate), _p(shared_w_up),
                            _p(shared_w_down), _p(y), _p(topk_idx), _p(topk_gate),
                            _p(counts_routed), _p(counts_kept), _p(aux), _p(ws),
                            ws.numel() if ws is not None else 0, _stream(stream)), "moe_forward")


def moe_forward_profiled(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate,
                         shared_w_up, shared_w_down, y, topk_idx, topk_gate, counts_routed,
                         counts_kept, aux, ws, events, stream=None):
    """moe_forward plus six torch.cuda.Event timestamps at the stage boundaries
    (before router, after router, after dispatch, after expert product 1, after
    expert product 2, after combine). Every event must have been recorded once
    before, so that its CUDA handle exists."""
    handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    _check(_lib.moe_forward_profiled(ctypes.byref(cfg), _p(x), _p(w_r), _p(b_r),
                                     _p(w_gate_or_w1), _p(w_up), _p(w_down), _p(shared_w_gate),
                                     _p(shared_w_up), _p(shared_w_down), _p(y), _p(topk_idx),
                                     _p(topk_gate), _p(counts_routed), _p(counts_kept), _p(aux),
                                     _p(ws), ws.numel() if ws is not None else 0,
                                     _stream(stream), handles, len(events)),
           "moe_forward_profiled")


class ForwardGraph:
    """Handle of a captured forward (moe_forward_graph_create). It keeps the tensors
    baked into the graph alive until destroy(); launch() enqueues one forward."""

    def __init__(self, handle, tensors, events):
        self.handle = handle
        self._keep = (tensors, events)

    def launch(self, stream=None):
        moe_forward_graph_launch(self, stream)

    def destroy(self):
        moe_forward_graph_destroy(self)

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            try:
                _lib.moe_forward_graph_destroy(h)
            except Exception:  # interpreter shutdown: the library may already be gone
                pass


def moe_forward_graph_create(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate,
                             shared_w_up, shared_w_down, y, topk_idx, topk_gate, counts_routed,
                             counts_kept, aux, ws, events=None) -> ForwardGraph:
    """Capture one moe_forward with these buffers into a CUDA graph. `events`: None or
    six torch.cuda.Event recorded at the stages (each recorded once before, so that its
    CUDA handle exists)."""
    tensors = (x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up,
               shared_w_down, y, topk_idx, topk_gate, counts_routed, counts_kept, aux, ws)
    handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events]) if events else None
    out = ctypes.c_void_p()
    _check(_lib.moe_forward_graph_create(ctypes.byref(cfg), *[_p(t) for t in tensors[:-1]], _p(ws),
                                         ws.numel() if ws is not None else 0, handles,
                                         len(events) if events else 0, ctypes.byref(out)),
           "moe_forward_graph_create")
    return ForwardGraph(out.value, tensors, events)


def moe_forward_graph_launch(graph, stream=None):
    h = graph.handle if isinstance(graph, ForwardGraph) else graph
    _check(_lib.moe_forward_graph_launch(h, _stream(stream)), "moe_forward_graph_launch")


def moe_forward_graph_destroy(graph):
    if isinstance(graph, ForwardGraph):
        h, graph.handle = graph.handle, None
    else:
        h = graph
    _check(_lib.moe_forward_graph_destroy(h), "moe_forward_graph_destroy")


def moe_check_error(ws, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns the status."""
    return _lib.moe_check_error(_p(ws), _stream(stream))


def library_path() -> str:
    return str(_LIB_PATH)
