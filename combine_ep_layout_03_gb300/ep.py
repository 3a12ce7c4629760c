"""Thin Python binding of libeplayout.so (the C ABI in include/ep_layout.h).

Argument marshalling only: torch tensors supply device memory and streams,
every step of layout / dispatch / combine runs in the library's CUDA kernels.
Importing this module loads the library and raises ImportError when it has not
been built (``python -m combine_ep_layout_03_gb300.build``); there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libeplayout.so")

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_CAPACITY = 0, 1, 2, 3
EP_ERR_BAD_EXPERT_ID, EP_ERR_TIMEOUT, EP_ERR_CUDA = 4, 5, 6

EP_QUANT_NONE = 0
EP_QUANT_INT8_STATIC = 1
EP_QUANT_INT8_PER_TOKEN = 2
EP_QUANT_MXFP8_E4M3 = 4
EP_QUANT_MXFP8_E5M2 = 5
EP_QUANT_MXFP4_E2M1 = 6
EP_QUANT_FP8_E4M3_PER_TOKEN = 7
EP_QUANT_FP8_E5M2_PER_TOKEN = 8
EP_QUANT_FP8_E4M3_PER_GROUP = 9
EP_QUANT_FP8_E5M2_PER_GROUP = 10
QUANT_MODES = (EP_QUANT_NONE, EP_QUANT_INT8_STATIC, EP_QUANT_INT8_PER_TOKEN, EP_QUANT_MXFP8_E4M3,
               EP_QUANT_MXFP8_E5M2, EP_QUANT_MXFP4_E2M1, EP_QUANT_FP8_E4M3_PER_TOKEN,
               EP_QUANT_FP8_E5M2_PER_TOKEN, EP_QUANT_FP8_E4M3_PER_GROUP, EP_QUANT_FP8_E5M2_PER_GROUP)

EP_SCALES_NONE, EP_SCALES_SCALAR, EP_SCALES_PER_CHANNEL, EP_SCALES_PER_EXPERT = 0, 1, 2, 3
# ep_dispatch_flag bits of ep_dispatch_ex
EP_DISPATCH_PER_RANK, EP_DISPATCH_SCALES_BLOCK_MAJOR, EP_DISPATCH_PRE_ENCODED = 1, 2, 4


class EPError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


class ep_params(ctypes.Structure):
    _fields_ = [("num_ranks", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("expert_alignment", ctypes.c_int32),
                ("recv_capacity_rows", ctypes.c_int64)]


class ep_layout_views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "cnt", "is_token_in_rank", "num_tokens_per_rank", "recv_cnt", "aligned_cnt",
        "expert_start", "rank_base", "expert_base", "src_prefix", "dst_row", "recv_src",
        "expert_ids", "expert_usage_stats")] + [("recv_src_capacity", ctypes.c_int64)] + [
        ("tok_dst", ctypes.c_void_p), ("recv_src_tok", ctypes.c_void_p),
        ("rank_tok_base", ctypes.c_void_p), ("tok_capacity", ctypes.c_int64)]


class ep_step_buffers(ctypes.Structure):
    _fields_ = [("topk", ctypes.c_void_p), ("weights", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("shared", ctypes.c_void_p), ("out", ctypes.c_void_p), ("recv_data", ctypes.c_void_p),
                ("recv_scales", ctypes.c_void_p), ("recv_rows_capacity", ctypes.c_int64),
                ("y", ctypes.c_void_p), ("y_rows_capacity", ctypes.c_int64)]


class ep_layout_outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "status", "cnt", "is_token_in_rank", "num_tokens_per_rank", "recv_cnt", "aligned_cnt",
        "expert_start", "rank_base", "expert_base", "src_prefix", "dst_row", "recv_src",
        "expert_ids", "expert_usage_stats")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libeplayout.so is not built ({LIB_PATH}); run "
                          "`python -m combine_ep_layout_03_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER(ep_params)
    sig = {
        "ep_status_string": ([st], ctypes.c_char_p),
        "ep_params_validate": ([P], st),
        "ep_layout_workspace_size": ([P, ctypes.POINTER(ctypes.c_size_t)], st),
        "ep_recv_row_bytes": ([i32, st, ctypes.POINTER(i64), ctypes.POINTER(i64)], st),
        "ep_handle_create": ([P, vp, ctypes.c_size_t, ctypes.POINTER(vp)], st),
        "ep_handle_destroy": ([vp], st),
        "ep_layout": ([vp, vp, vp], st),
        "ep_layout_masked": ([vp, vp, vp, i32, vp], st),
        "ep_handle_views": ([vp, ctypes.POINTER(ep_layout_views)], st),
        "ep_handle_recv_rows": ([vp, vp, vp], st),
        "ep_handle_expert_counts": ([vp, vp, vp], st),
        "ep_handle_status": ([vp, vp], st),
        "ep_dispatch": ([vp, vp, st, vp, vp, i64, vp], st),
        "ep_dispatch_scaled": ([vp, vp, st, vp, st, vp, vp, i64, vp], st),
        "ep_combine": ([vp, vp, i64, vp, vp, i32, vp, vp], st),
        "ep_expert_identity": ([vp, st, vp, vp, i64, i32, vp, vp], st),
        "ep_layout_static_scratch": ([P, vp, ctypes.POINTER(ep_layout_outputs), vp], st),
        "ep_token_layout": ([vp, vp, vp, vp, i32, vp, vp, i64, vp], st),
        "ep_handle_token_rows": ([vp, vp, vp], st),
        "ep_dispatch_tokens": ([vp, vp, st, vp, st, vp, vp, i64, vp], st),
        "ep_combine_tokens": ([vp, vp, i64, vp, i32, vp, vp, vp, vp], st),
        "ep_expert_identity_tokens": ([vp, st, vp, vp, vp, vp, i64, i32, vp, vp], st),
        "ep_dispatch_ex": ([vp, vp, vp, st, vp, st, ctypes.c_uint32, vp, vp, i64, vp], st),
        "ep_combine_add_rms_norm": ([vp, vp, i64, vp, vp, i32, vp, vp, ctypes.c_float, vp, vp, vp, vp], st),
        "ep_test_combine_stalled": ([vp, vp, i64, vp, vp, ctypes.c_uint32, vp], st),
        "ep_step_host": ([vp, st, vp, vp, vp, vp, i32, vp, ctypes.POINTER(ep_step_buffers), vp], st),
        "ep_dispatch_async": ([vp, vp, st, vp, st, vp, vp, i64, vp], st),
        "ep_dispatch_wait": ([vp, st, vp, vp, i64, ctypes.c_uint32, vp, vp, i64, vp], st),
        "ep_combine_async": ([vp, vp, i64, vp, i64, vp], st),
        "ep_combine_wait": ([vp, vp, i64, vp, vp, i32, vp, vp], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()
lib = _lib


def status_string(status: int) -> str:
    return _lib.ep_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != EP_OK:
        raise EPError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_params(R, T, H, E, K, alpha=1, recv_capacity_rows=0) -> ep_params:
    return ep_params(R, T, H, E, K, alpha, recv_capacity_rows)


# ---------------------------------------------------------------- C-named calls

def ep_params_validate(p: ep_params) -> int:
    return _lib.ep_params_validate(ctypes.byref(p))


def ep_layout_workspace_size(p: ep_params) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.ep_layout_workspace_size(ctypes.byref(p), ctypes.byref(n)), "ep_layout_workspace_size")
    return int(n.value)


def ep_recv_row_bytes(hidden: int, quant: int) -> tuple[int, int]:
    d, s = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(_lib.ep_recv_row_bytes(hidden, quant, ctypes.byref(d), ctypes.byref(s)), "ep_recv_row_bytes")
    return int(d.value), int(s.value)


def ep_handle_create(p: ep_params, workspace: torch.Tensor) -> int:
    h = ctypes.c_void_p(0)
    _check(_lib.ep_handle_create(ctypes.byref(p), workspace.data_ptr(), workspace.numel(),
                                 ctypes.byref(h)), "ep_handle_create")
    return int(h.value)


def ep_handle_destroy(h: int) -> None:
    _lib.ep_handle_destroy(h)


def ep_layout(h: int, topk_idx: torch.Tensor, stream=None) -> None:
    _check(_lib.ep_layout(h, _ptr(topk_idx), _stream(stream)), "ep_layout")


def ep_layout_masked(h: int, topk_idx: torch.Tensor, mask, mask_dims: int, stream=None) -> None:
    _check(_lib.ep_layout_masked(h, _ptr(topk_idx), _ptr(mask), int(mask_dims), _stream(stream)),
           "ep_layout_masked")


def ep_handle_views(h: int) -> ep_layout_views:
    v = ep_layout_views()
    _check(_lib.ep_handle_views(h, ctypes.byref(v)), "ep_handle_views")
    return v


def ep_handle_recv_rows(h: int, R: int, stream=None) -> list[int]:
    buf = (ctypes.c_int64 * (R + 1))()
    _check(_lib.ep_handle_recv_rows(h, ctypes.addressof(buf), _stream(stream)), "ep_handle_recv_rows")
    return list(buf)


def ep_handle_expert_counts(h: int, E: int, stream=None) -> list[int]:
    buf = (ctypes.c_int32 * E)()
    _check(_lib.ep_handle_expert_counts(h, ctypes.addressof(buf), _stream(stream)),
           "ep_handle_expert_counts")
    return list(buf)


def ep_handle_status(h: int, stream=None) -> int:
    return int(_lib.ep_handle_status(h, _stream(stream)))


def ep_dispatch(h: int, x, quant: int, recv_data, recv_scales, recv_rows_capacity: int,
                stream=None) -> None:
    _check(_lib.ep_dispatch(h, _ptr(x), quant, _ptr(recv_data), _ptr(recv_scales),
                            int(recv_rows_capacity), _stream(stream)), "ep_dispatch")


def ep_dispatch_scaled(h: int, x, quant: int, scales, scale_kind: int, recv_data, recv_scales,
                       recv_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_dispatch_scaled(h, _ptr(x), quant, _ptr(scales), int(scale_kind), _ptr(recv_data),
                                   _ptr(recv_scales), int(recv_rows_capacity), _stream(stream)),
           "ep_dispatch_scaled")


def ep_dispatch_ex(h: int, x, x_scales, quant: int, scales, scale_kind: int, flags: int, recv_data,
                   recv_scales, recv_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_dispatch_ex(h, _ptr(x), _ptr(x_scales), quant, _ptr(scales), int(scale_kind),
                               int(flags), _ptr(recv_data), _ptr(recv_scales), int(recv_rows_capacity),
                               _stream(stream)), "ep_dispatch_ex")


def ep_combine_add_rms_norm(h: int, y, y_rows_capacity: int, topk_weights, shared, num_shared: int,
                            residual, gamma, eps: float, norm_out, x_out, rstd_out, stream=None) -> None:
    _check(_lib.ep_combine_add_rms_norm(h, _ptr(y), int(y_rows_capacity), _ptr(topk_weights), _ptr(shared),
                                        int(num_shared), _ptr(residual), _ptr(gamma), float(eps),
                                        _ptr(norm_out), _ptr(x_out), _ptr(rstd_out), _stream(stream)),
           "ep_combine_add_rms_norm")


def step_buffers(topk, weights, x, out, recv_data, recv_scales=None, shared=None, y=None,
                 H: int | None = None) -> ep_step_buffers:
    """ep_step_buffers from device tensors (capacities from their sizes)."""
    b = ep_step_buffers()
    b.topk, b.weights, b.x, b.out = _ptr(topk), _ptr(weights), _ptr(x), _ptr(out)
    b.shared, b.recv_data, b.recv_scales, b.y = _ptr(shared), _ptr(recv_data), _ptr(recv_scales), _ptr(y)
    b.recv_rows_capacity = recv_data.shape[0]
    b.y_rows_capacity = 0 if y is None else y.numel() // (H or y.shape[-1])
    return b


def ep_step_host(h: int, quant: int, topk_host, weights_host, x_host, shared_host, num_shared: int, out_host,
                 bufs: ep_step_buffers, stream=None) -> None:
    """One step from (pinned) host tensors: copy in, layout, dispatch, combine, copy out."""
    _check(_lib.ep_step_host(h, quant, _ptr(topk_host), _ptr(weights_host), _ptr(x_host), _ptr(shared_host),
                             int(num_shared), _ptr(out_host), ctypes.byref(bufs), _stream(stream)), "ep_step_host")


def ep_test_combine_stalled(h: int, y, y_rows_capacity: int, topk_weights, out, max_polls: int,
                            stream=None) -> None:
    """Test hook: the combine with a producer that issues nothing (bounded waits run out)."""
    _check(_lib.ep_test_combine_stalled(h, _ptr(y), int(y_rows_capacity), _ptr(topk_weights), _ptr(out),
                                        int(max_polls), _stream(stream)), "ep_test_combine_stalled")


def ep_dispatch_async(h: int, x, quant: int, scales, scale_kind: int, tok_data, tok_scales,
                      tok_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_dispatch_async(h, _ptr(x), quant, _ptr(scales), int(scale_kind), _ptr(tok_data),
                                  _ptr(tok_scales), int(tok_rows_capacity), _stream(stream)), "ep_dispatch_async")


def ep_dispatch_wait(h: int, quant: int, tok_data, tok_scales, tok_rows_capacity: int, flags: int, recv_data,
                     recv_scales, recv_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_dispatch_wait(h, quant, _ptr(tok_data), _ptr(tok_scales), int(tok_rows_capacity), int(flags),
                                 _ptr(recv_data), _ptr(recv_scales), int(recv_rows_capacity), _stream(stream)),
           "ep_dispatch_wait")


def ep_combine_async(h: int, y, y_rows_capacity: int, ret, ret_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_combine_async(h, _ptr(y), int(y_rows_capacity), _ptr(ret), int(ret_rows_capacity),
                                 _stream(stream)), "ep_combine_async")


def ep_combine_wait(h: int, ret, ret_rows_capacity: int, topk_weights, shared, num_shared: int, out,
                    stream=None) -> None:
    _check(_lib.ep_combine_wait(h, _ptr(ret), int(ret_rows_capacity), _ptr(topk_weights), _ptr(shared),
                                int(num_shared), _ptr(out), _stream(stream)), "ep_combine_wait")


def ep_combine(h: int, y, y_rows_capacity: int, topk_weights, shared, num_shared: int, out,
               stream=None) -> None:
    _check(_lib.ep_combine(h, _ptr(y), int(y_rows_capacity), _ptr(topk_weights), _ptr(shared),
                           int(num_shared), _ptr(out), _stream(stream)), "ep_combine")


def ep_expert_identity(h: int, quant: int, recv_data, recv_scales, rows_capacity: int,
                       mark_mod: int, y, stream=None) -> None:
    _check(_lib.ep_expert_identity(h, quant, _ptr(recv_data), _ptr(recv_scales),
                                   int(rows_capacity), int(mark_mod), _ptr(y), _stream(stream)),
           "ep_expert_identity")


def ep_token_layout(h: int, topk_idx, topk_weights, mask, mask_dims: int, recv_topk_idx,
                    recv_topk_weights, rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_token_layout(h, _ptr(topk_idx), _ptr(topk_weights), _ptr(mask), int(mask_dims),
                                _ptr(recv_topk_idx), _ptr(recv_topk_weights), int(rows_capacity),
                                _stream(stream)), "ep_token_layout")


def ep_handle_token_rows(h: int, R: int, stream=None) -> list[int]:
    buf = (ctypes.c_int64 * (R + 1))()
    _check(_lib.ep_handle_token_rows(h, ctypes.addressof(buf), _stream(stream)), "ep_handle_token_rows")
    return list(buf)


def ep_dispatch_tokens(h: int, x, quant: int, scales, scale_kind: int, recv_data, recv_scales,
                       recv_rows_capacity: int, stream=None) -> None:
    _check(_lib.ep_dispatch_tokens(h, _ptr(x), quant, _ptr(scales), int(scale_kind), _ptr(recv_data),
                                   _ptr(recv_scales), int(recv_rows_capacity), _stream(stream)),
           "ep_dispatch_tokens")


def ep_combine_tokens(h: int, y, y_rows_capacity: int, shared, num_shared: int, out, rank_weights,
                      out_weights, stream=None) -> None:
    _check(_lib.ep_combine_tokens(h, _ptr(y), int(y_rows_capacity), _ptr(shared), int(num_shared),
                                  _ptr(out), _ptr(rank_weights), _ptr(out_weights), _stream(stream)),
           "ep_combine_tokens")


def ep_expert_identity_tokens(h: int, quant: int, recv_data, recv_scales, recv_topk_idx,
                              recv_topk_weights, rows_capacity: int, mark_mod: int, y,
                              stream=None) -> None:
    _check(_lib.ep_expert_identity_tokens(h, quant, _ptr(recv_data), _ptr(recv_scales),
                                          _ptr(recv_topk_idx), _ptr(recv_topk_weights),
                                          int(rows_capacity), int(mark_mod), _ptr(y), _stream(stream)),
           "ep_expert_identity_tokens")


# ---------------------------------------------------------------- convenience wrapper

_VIEW_SPECS = {
    # name: (dtype, shape builder)
    "cnt": (torch.int32, lambda s: (s.R, s.E)),
    "is_token_in_rank": (torch.uint8, lambda s: (s.R, s.T, s.R)),
    "num_tokens_per_rank": (torch.int32, lambda s: (s.R, s.R)),
    "recv_cnt": (torch.int32, lambda s: (s.E,)),
    "aligned_cnt": (torch.int32, lambda s: (s.R, s.L)),
    "expert_start": (torch.int32, lambda s: (s.R, s.L + 1)),
    "rank_base": (torch.int64, lambda s: (s.R + 1,)),
    "expert_base": (torch.int32, lambda s: (s.E + 1,)),
    "src_prefix": (torch.int32, lambda s: (s.R, s.E)),
    "dst_row": (torch.int32, lambda s: (s.R, s.T, s.K)),
    "recv_src": (torch.int32, lambda s: (s.recv_src_capacity,)),
    "expert_ids": (torch.int32, lambda s: (s.R, s.L)),
    "expert_usage_stats": (torch.int32, lambda s: (s.R, 2)),
    "tok_dst": (torch.int32, lambda s: (s.R, s.T, s.K)),
    "recv_src_tok": (torch.int32, lambda s: (s.tok_capacity,)),
    "rank_tok_base": (torch.int64, lambda s: (s.R + 1,)),
}


class EPLayout:
    """A handle plus its device workspace (a torch uint8 tensor).

    ``layout(topk_idx)`` fills the handle; ``views()`` exposes the layout arrays
    as torch tensors aliasing the workspace; ``dispatch`` / ``combine`` run the
    kernels on caller tensors.  R logical ranks share one GPU."""

    def __init__(self, R, T, H, E, K, alpha=1, recv_capacity_rows=0, device="cuda"):
        self.R, self.T, self.H, self.E, self.K, self.alpha = R, T, H, E, K, alpha
        self.L = E // R
        self.params = make_params(R, T, H, E, K, alpha, recv_capacity_rows)
        nbytes = ep_layout_workspace_size(self.params)
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.workspace.data_ptr()) % 256
        self.ws = self.workspace[off:off + nbytes]
        self.h = ep_handle_create(self.params, self.ws)
        v = ep_handle_views(self.h)
        self.recv_src_capacity = v.recv_src_capacity
        self.tok_capacity = v.tok_capacity

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            ep_handle_destroy(h)
            self.h = None

    @property
    def worst_rows(self) -> int:
        return self.R * self.T * self.K + self.E * (self.alpha - 1)

    def layout(self, topk_idx: torch.Tensor, stream=None, active_mask: torch.Tensor | None = None
               ) -> "EPLayout":
        """active_mask (xActiveMask): uint8/bool [R, T] per token or [R, T, K] per entry."""
        assert topk_idx.dtype == torch.int64 and topk_idx.is_contiguous()
        assert topk_idx.numel() == self.R * self.T * self.K
        if active_mask is None:
            ep_layout(self.h, topk_idx, stream)
        else:
            m = active_mask.to(torch.uint8).contiguous()
            dims = 1 if m.numel() == self.R * self.T else 2
            assert m.numel() == (self.R * self.T if dims == 1 else self.R * self.T * self.K)
            self._mask = m  # keep alive until the kernels ran
            ep_layout_masked(self.h, topk_idx, m, dims, stream)
        return self

    def views(self) -> dict[str, torch.Tensor]:
        v = ep_handle_views(self.h)
        base = self.ws.data_ptr()
        out = {}
        for name, (dt, shape) in _VIEW_SPECS.items():
            shp = shape(self)
            n = 1
            for d in shp:
                n *= d
            off = getattr(v, name) - base
            nbytes = n * torch.empty((), dtype=dt).element_size()
            out[name] = self.ws[off:off + nbytes].view(dt).view(shp)
        return out

    def recv_rows(self, stream=None) -> list[int]:
        """rank_base on the host (synchronises the stream)."""
        return ep_handle_recv_rows(self.h, self.R, stream)

    def expert_counts(self, stream=None) -> list[int]:
        return ep_handle_expert_counts(self.h, self.E, stream)

    def status(self, stream=None) -> int:
        return ep_handle_status(self.h, stream)

    def alloc_recv(self, quant: int, rows: int | None = None, device="cuda"):
        rows = self.worst_rows if rows is None else rows
        db, sb = ep_recv_row_bytes(self.H, quant)
        data = torch.empty((rows, db), dtype=torch.uint8, device=device)
        scales = torch.empty((rows, sb), dtype=torch.uint8, device=device) if sb else None
        return data, scales

    def dispatch(self, x: torch.Tensor, quant: int, recv_data: torch.Tensor,
                 recv_scales: torch.Tensor | None, stream=None, scales: torch.Tensor | None = None,
                 scale_kind: int = EP_SCALES_NONE) -> None:
        db, _ = ep_recv_row_bytes(self.H, quant)
        cap = recv_data.numel() // db
        if scales is None and scale_kind == EP_SCALES_NONE:
            ep_dispatch(self.h, x, quant, recv_data, recv_scales, cap, stream)
        else:
            ep_dispatch_scaled(self.h, x, quant, scales, scale_kind, recv_data, recv_scales, cap, stream)

    def alloc_recv_block_major(self, quant: int, rows: int, device="cuda"):
        """Receive buffers whose scales are block-major: (blocks, rows) elements,
        uint8 [blocks, rows * element bytes]."""
        db, sb = ep_recv_row_bytes(self.H, quant)
        es = 1 if quant in (EP_QUANT_MXFP8_E4M3, EP_QUANT_MXFP8_E5M2, EP_QUANT_MXFP4_E2M1) else 4
        data = torch.empty((rows, db), dtype=torch.uint8, device=device)
        scales = torch.empty((sb // es, rows * es), dtype=torch.uint8, device=device) if sb else None
        return data, scales

    def dispatch_ex(self, x: torch.Tensor, quant: int, recv_data: torch.Tensor,
                    recv_scales: torch.Tensor | None, stream=None, *, x_scales=None, scales=None,
                    scale_kind: int = EP_SCALES_NONE, per_rank: bool = False,
                    block_major: bool = False, pre_encoded: bool = False) -> None:
        """ep_dispatch_ex: pre_encoded moves (x, x_scales) byte rows unchanged;
        block_major writes the scales (blocks, capacity)."""
        db, _ = ep_recv_row_bytes(self.H, quant)
        flags = ((EP_DISPATCH_PER_RANK if per_rank else 0) |
                 (EP_DISPATCH_SCALES_BLOCK_MAJOR if block_major else 0) |
                 (EP_DISPATCH_PRE_ENCODED if pre_encoded else 0))
        ep_dispatch_ex(self.h, x, x_scales, quant, scales, scale_kind, flags, recv_data, recv_scales,
                       recv_data.numel() // db, stream)

    def combine(self, y: torch.Tensor, topk_weights: torch.Tensor, out: torch.Tensor,
                shared: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        S = 0 if shared is None else shared.shape[1]
        cap = y.numel() // self.H
        ep_combine(self.h, y, cap, topk_weights, shared, S, out, stream)
        return out

    def dispatch_async(self, x, quant, tok_data, tok_scales, stream=None, scales=None,
                       scale_kind=EP_SCALES_NONE) -> None:
        """Send phase: rows into the per-rank arrival layout (after token_layout)."""
        db, _ = ep_recv_row_bytes(self.H, quant)
        ep_dispatch_async(self.h, x, quant, scales, scale_kind, tok_data, tok_scales, tok_data.numel() // db,
                          stream)

    def dispatch_wait(self, quant, tok_data, tok_scales, recv_data, recv_scales, stream=None,
                      block_major: bool = False) -> None:
        """Wait phase: arrival rows -> per-expert grouped rows."""
        db, _ = ep_recv_row_bytes(self.H, quant)
        ep_dispatch_wait(self.h, quant, tok_data, tok_scales, tok_data.numel() // db,
                         EP_DISPATCH_SCALES_BLOCK_MAJOR if block_major else 0, recv_data, recv_scales,
                         recv_data.numel() // db, stream)

    def alloc_return(self, device="cuda") -> torch.Tensor:
        """Token-major return buffer of the two-phase combine, [R*T*K, H] bf16."""
        return torch.empty((max(self.R * self.T * self.K, 1), self.H), dtype=torch.bfloat16, device=device)

    def combine_async(self, y: torch.Tensor, ret: torch.Tensor, stream=None) -> None:
        ep_combine_async(self.h, y, y.numel() // self.H, ret, ret.numel() // self.H, stream)

    def combine_wait(self, ret: torch.Tensor, topk_weights: torch.Tensor, out: torch.Tensor,
                     shared: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        S = 0 if shared is None else shared.shape[1]
        ep_combine_wait(self.h, ret, ret.numel() // self.H, topk_weights, shared, S, out, stream)
        return out

    def combine_add_rms_norm(self, y: torch.Tensor, topk_weights: torch.Tensor, residual: torch.Tensor,
                             gamma: torch.Tensor, norm_out: torch.Tensor, x_out: torch.Tensor | None = None,
                             rstd_out: torch.Tensor | None = None, shared: torch.Tensor | None = None,
                             eps: float = 1e-6, stream=None) -> torch.Tensor:
        """Combine, then x = combine + residual and norm_out = RMSNorm(x) * gamma."""
        S = 0 if shared is None else shared.shape[1]
        ep_combine_add_rms_norm(self.h, y, y.numel() // self.H, topk_weights, shared, S, residual, gamma,
                                eps, norm_out, x_out, rstd_out, stream)
        return norm_out

    def expert_identity(self, quant: int, recv_data, recv_scales, y, mark_mod: int = 0,
                        stream=None) -> torch.Tensor:
        db, _ = ep_recv_row_bytes(self.H, quant)
        cap = min(recv_data.numel() // db, y.numel() // self.H)
        ep_expert_identity(self.h, quant, recv_data, recv_scales, cap, mark_mod, y, stream)
        return y

    # ---------------------------------------------------------- per-rank layout

    def token_layout(self, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                     active_mask: torch.Tensor | None = None, rows_capacity: int | None = None,
                     stream=None, out=None):
        """DeepEP per-rank receive layout; call after layout() with the same topk and
        mask.  Returns (recv_topk_idx [cap, K] int64, recv_topk_weights [cap, K] f32),
        written into ``out`` when given."""
        dev = topk_idx.device
        if out is not None:
            ridx, rw = out
            cap = ridx.shape[0] if rows_capacity is None else rows_capacity
        else:
            cap = self.tok_capacity if rows_capacity is None else rows_capacity
            ridx = torch.empty((max(cap, 1), self.K), dtype=torch.int64, device=dev)
            rw = torch.empty((max(cap, 1), self.K), dtype=torch.float32, device=dev)
        m, dims = None, 0
        if active_mask is not None:
            m = active_mask.to(torch.uint8).contiguous()
            dims = 1 if m.numel() == self.R * self.T else 2
            self._tmask = m
        ep_token_layout(self.h, topk_idx, topk_weights.contiguous(), m, dims, ridx, rw, cap, stream)
        return ridx, rw

    def token_rows(self, stream=None) -> list[int]:
        return ep_handle_token_rows(self.h, self.R, stream)

    def dispatch_tokens(self, x, quant, recv_data, recv_scales, stream=None, scales=None,
                        scale_kind=EP_SCALES_NONE) -> None:
        db, _ = ep_recv_row_bytes(self.H, quant)
        ep_dispatch_tokens(self.h, x, quant, scales, scale_kind, recv_data, recv_scales,
                           recv_data.numel() // db, stream)

    def combine_tokens(self, y, out, shared=None, rank_weights=None, out_weights=None, stream=None):
        S = 0 if shared is None else shared.shape[1]
        ep_combine_tokens(self.h, y, y.numel() // self.H, shared, S, out, rank_weights, out_weights,
                          stream)
        return out

    def expert_identity_tokens(self, quant, recv_data, recv_scales, recv_topk_idx, recv_topk_weights,
                               y, mark_mod: int = 0, stream=None):
        db, _ = ep_recv_row_bytes(self.H, quant)
        cap = min(recv_data.numel() // db, y.numel() // self.H, recv_topk_idx.shape[0])
        ep_expert_identity_tokens(self.h, quant, recv_data, recv_scales, recv_topk_idx,
                                  recv_topk_weights, cap, mark_mod, y, stream)
        return y


def ep_layout_static_scratch(p: ep_params, topk_idx, outputs: dict, stream=None) -> None:
    """The layout without any device allocation: ``outputs`` maps each field of
    ep_layout_outputs to a caller-owned device tensor (or pointer)."""
    o = ep_layout_outputs(**{k: _ptr(outputs[k]) for k, _ in ep_layout_outputs._fields_})
    _check(_lib.ep_layout_static_scratch(ctypes.byref(p), _ptr(topk_idx), ctypes.byref(o),
                                         _stream(stream)), "ep_layout_static_scratch")
