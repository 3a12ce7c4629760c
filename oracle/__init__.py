"""CPU oracle for the MoE expert-parallel layout -> dispatch -> combine path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA path (``combine_ep_layout_03_gb300``) and never imports it.

The arithmetic lives in ``ep_oracle.c`` (plain C, compiled here with gcc, no
FMA contraction, no fast-math); this module only marshals numpy arrays.  Each
wrapped function cites, in the C source, the passage of the pages it follows:
the DeepEP "Normal Mode API" (dispatch/combine parameters and returns), CANN
"aclnnMoeDistributeDispatchV2" (Formula section: quantMode 0, 2 and 4) and
Modular MAX "EPBatchManager" (ep_dispatch outputs, ep_combine).

Parity pins: every function here is pinned by the CPU tests in
``tests/test_oracle_*.py`` against brute force, closed forms, library
routines and hand-worked rows.  Two readings are not fixed by any value on the
pages and are marked "parity unpinned": the e8m0 byte stores the decode scale
2^sharedExp (not its inverse), and e2m1 packs element 2i in the low nibble.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libeporacle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

# quant-mode numbers of the C-ABI enum
Q_NONE, Q_INT8_STATIC, Q_INT8, Q_E4M3, Q_E5M2, Q_E2M1 = 0, 1, 2, 4, 5, 6
Q_FP8T_E4M3, Q_FP8T_E5M2, Q_FP8G_E4M3, Q_FP8G_E5M2 = 7, 8, 9, 10
QUANT_MODES = (Q_NONE, Q_INT8_STATIC, Q_INT8, Q_E4M3, Q_E5M2, Q_E2M1,
               Q_FP8T_E4M3, Q_FP8T_E5M2, Q_FP8G_E4M3, Q_FP8G_E5M2)
# kinds of the input scales of quantModes 1-3
S_NONE, S_SCALAR, S_CHANNEL, S_EXPERT = 0, 1, 2, 3
GROUP = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc).  Returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if path is not None:
            return _declare(ctypes.CDLL(path))
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _declare(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
    lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_mini_encode.argtypes = [i32, ctypes.c_float]
    lib.oracle_mini_encode.restype = i32
    lib.oracle_mini_decode.argtypes = [i32, i32]
    lib.oracle_mini_decode.restype = ctypes.c_double
    lib.oracle_quant_int8_row.argtypes = [i32, vp, vp, vp]
    lib.oracle_quant_mx_row.argtypes = [i32, i32, vp, vp, vp]
    lib.oracle_row_data_bytes.argtypes = [i32, i32]
    lib.oracle_row_data_bytes.restype = i64
    lib.oracle_row_scale_bytes.argtypes = [i32, i32]
    lib.oracle_row_scale_bytes.restype = i64
    lib.oracle_layout.argtypes = [i32, i32, i32, i32, i32, vp, i64] + [vp] * 12
    lib.oracle_layout.restype = i32
    lib.oracle_dispatch.argtypes = [i32, i32, i32, i32, vp, vp, i64, i64, vp, vp]
    lib.oracle_dispatch_rows.argtypes = [i64, vp, vp, i32, i32, vp, vp, vp]
    lib.oracle_expert_rows.argtypes = [i64, vp, vp, i32, i32, vp, vp, i32, vp]
    lib.oracle_combine.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, i64, vp]
    lib.oracle_combine_ref64.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, i64, vp, vp]
    lib.oracle_quant_fp8_token_row.argtypes = [i32, i32, vp, vp, vp, vp]
    lib.oracle_quant_fp8_group_row.argtypes = [i32, i32, vp, vp, vp, vp]
    lib.oracle_quant_int8_static_row.argtypes = [i32, vp, vp, vp]
    lib.oracle_quant_int8_row_scaled.argtypes = [i32, vp, vp, vp, vp]
    lib.oracle_encode_row_scaled.argtypes = [i32, i32, vp, vp, vp, vp]
    lib.oracle_dispatch_scaled.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, i32, i64, i64, vp, vp]
    lib.oracle_layout_masked.argtypes = [i32, i32, i32, i32, i32, vp, vp, i32, i64] + [vp] * 12
    lib.oracle_layout_masked.restype = i32
    lib.oracle_token_layout.argtypes = [i32, i32, i32, i32, vp, vp, i64, vp, vp, vp, vp, vp]
    lib.oracle_token_layout.restype = i64
    lib.oracle_expert_token_rows.argtypes = [i64, vp, i32, i32, i32, vp, vp, vp, vp, i32, vp]
    lib.oracle_reduce_token_weights.argtypes = [i64, i32, vp, vp, vp]
    lib.oracle_dispatch_bytes.argtypes = [i32, i32, vp, vp, i64, i64, i64, vp]
    lib.oracle_encode_row.argtypes = [i32, i32, vp, vp, vp]
    lib.oracle_encode_rows.argtypes = [i32, i32, i64, vp, vp, vp]
    lib.oracle_add_rms_norm_ref64.argtypes = [i64, i32, vp, vp, vp, ctypes.c_double, vp, vp, vp]
    lib.oracle_add_rms_norm_f32.argtypes = [i64, i32, vp, vp, vp, ctypes.c_float, vp, vp, vp]
    return lib


# ---------------------------------------------------------------------------
# scalar encoders
# ---------------------------------------------------------------------------

def bf16_from_f32(values) -> np.ndarray:
    lib = load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_bf16_from_f32(float(x)) for x in v], dtype=np.uint16)


def mini_encode(q: int, values) -> np.ndarray:
    lib = load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_mini_encode(q, float(x)) for x in v], dtype=np.int32)


def mini_decode(q: int, codes) -> np.ndarray:
    lib = load()
    return np.array([lib.oracle_mini_decode(q, int(c)) for c in np.asarray(codes).ravel()])


def row_bytes(q: int, H: int) -> tuple[int, int]:
    lib = load()
    return int(lib.oracle_row_data_bytes(q, H)), int(lib.oracle_row_scale_bytes(q, H))


# ---------------------------------------------------------------------------
# quantisation of single rows
# ---------------------------------------------------------------------------

def quant_int8_row(x_bf16: np.ndarray) -> tuple[np.ndarray, np.float32]:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    q = np.zeros(x.shape[-1], dtype=np.int8)
    inv = np.zeros(1, dtype=np.float32)
    load().oracle_quant_int8_row(x.shape[-1], _p(x), _p(q), _p(inv))
    return q, inv[0]


def quant_mx_row(q: int, x_bf16: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    db, sb = row_bytes(q, H)
    codes = np.zeros(db, dtype=np.uint8)
    scales = np.zeros(sb, dtype=np.uint8)
    load().oracle_quant_mx_row(H, q, _p(x), _p(codes), _p(scales))
    return codes, scales


def _scale_arr(smooth, H):
    return None if smooth is None else np.ascontiguousarray(np.broadcast_to(
        np.asarray(smooth, np.float32), (H,)), dtype=np.float32)


def quant_fp8_token_row(fp8: int, x_bf16: np.ndarray, smooth=None):
    """Per-token FP8 (quantMode 2, FP8 destination): (codes [H] u8, inv f32)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    codes = np.zeros(H, np.uint8)
    inv = np.zeros(1, np.float32)
    sm = _scale_arr(smooth, H)
    load().oracle_quant_fp8_token_row(H, fp8, _p(x), _p(sm), _p(codes), _p(inv))
    return codes, inv[0]


def quant_fp8_group_row(fp8: int, x_bf16: np.ndarray, smooth=None):
    """Per-group-128 FP8 (quantMode 3): (codes [H] u8, inv [H/128] f32)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    codes = np.zeros(H, np.uint8)
    inv = np.zeros(H // GROUP, np.float32)
    sm = _scale_arr(smooth, H)
    load().oracle_quant_fp8_group_row(H, fp8, _p(x), _p(sm), _p(codes), _p(inv))
    return codes, inv


def quant_int8_static_row(x_bf16: np.ndarray, smooth) -> np.ndarray:
    """Static int8 (quantMode 1): codes of x * scales, saturated to [-128, 127]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    q = np.zeros(H, np.int8)
    load().oracle_quant_int8_static_row(H, _p(x), _p(_scale_arr(smooth, H)), _p(q))
    return q


def encode_row(q: int, x_bf16: np.ndarray, smooth=None):
    """Receive-row bytes (data, scale) of one source row, optional smooth scales."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    db, sb = row_bytes(q, H)
    data = np.zeros(db, np.uint8)
    scale = np.zeros(max(sb, 1), np.uint8)
    if smooth is None:
        load().oracle_encode_row(q, H, _p(x), _p(data), _p(scale))
    else:
        assert q in (Q_INT8_STATIC, Q_INT8, Q_FP8T_E4M3, Q_FP8T_E5M2, Q_FP8G_E4M3, Q_FP8G_E5M2)
        load().oracle_encode_row_scaled(q, H, _p(x), _p(_scale_arr(smooth, H)), _p(data), _p(scale))
    return data, scale[:sb]


def encode_rows(q: int, x_bf16: np.ndarray, threads: int = 1):
    """Receive-row bytes (data [n, db], scales [n, sb]) of every source row of
    x [n, H], each encoded once (the per-token encoding of dispatch).  With
    threads > 1, contiguous chunks of rows are encoded on that many threads at
    once (the C calls release the interpreter lock and share no state)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    H = x.shape[-1]
    x = x.reshape(-1, H)
    n = x.shape[0]
    db, sb = row_bytes(q, H)
    data = np.empty((n, db), np.uint8)
    scales = np.empty((n, sb), np.uint8)
    lib = load()

    def part(a, b):
        if b > a:
            lib.oracle_encode_rows(q, H, b - a, _p(x[a:b]), _p(data[a:b]), _p(scales[a:b]) if sb else None)

    if threads <= 1 or n < 2 * threads:
        part(0, n)
    else:
        from concurrent.futures import ThreadPoolExecutor
        step = -(-n // threads)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda a: part(a, min(n, a + step)), range(0, n, step)))
    return data, scales


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------

class Layout:
    """Result of :func:`layout` (numpy arrays, shapes as in the C source)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)

    @property
    def rows(self) -> int:
        return int(self.rank_base[-1])


def layout(R: int, T: int, E: int, K: int, alpha: int, topk: np.ndarray,
           recv_cap: int | None = None, mask: np.ndarray | None = None) -> Layout:
    """Layout of topk; mask (xActiveMask) is [R, T] (1-D per token) or
    [R, T, K] (2-D per entry), nonzero = active, or None."""
    topk = np.ascontiguousarray(topk, dtype=np.int64).reshape(R * T * K)
    L = E // R
    if recv_cap is None:
        recv_cap = R * T * K + E * (alpha - 1)
    out = dict(
        cnt=np.zeros((R, E), np.int32),
        is_token_in_rank=np.zeros((R, T, R), np.uint8),
        num_tokens_per_rank=np.zeros((R, R), np.int32),
        recv_cnt=np.zeros(E, np.int32),
        aligned=np.zeros(E, np.int32),
        expert_start=np.zeros((R, L + 1), np.int32),
        rank_base=np.zeros(R + 1, np.int64),
        src_prefix=np.zeros((R, E), np.int32),
        dst_row=np.zeros((R, T, K), np.int32),
        recv_src=np.full(max(recv_cap, 1), -1, np.int32),
        expert_ids=np.zeros((R, L), np.int32),
        expert_usage_stats=np.zeros((R, 2), np.int32),
    )
    outs = (_p(out[k]) for k in ("cnt", "is_token_in_rank", "num_tokens_per_rank", "recv_cnt",
                                 "aligned", "expert_start", "rank_base", "src_prefix", "dst_row",
                                 "recv_src", "expert_ids", "expert_usage_stats"))
    if mask is None:
        st = load().oracle_layout(R, T, E, K, alpha, _p(topk), recv_cap, *outs)
    else:
        m = np.ascontiguousarray(mask, dtype=np.uint8)
        dims = 1 if m.size == R * T else 2
        assert m.size == (R * T if dims == 1 else R * T * K)
        st = load().oracle_layout_masked(R, T, E, K, alpha, _p(topk), _p(m), dims, recv_cap, *outs)
    rows = int(out["rank_base"][-1])
    out["recv_src"] = out["recv_src"][: min(rows, recv_cap)]
    return Layout(status=int(st), R=R, T=T, E=E, K=K, alpha=alpha, L=L, **out)


def row_expert(lay: Layout) -> np.ndarray:
    """Expert id of every receive row (padding rows included)."""
    e = np.repeat(np.arange(lay.E, dtype=np.int32), lay.aligned.astype(np.int64))
    return e.astype(np.int32)


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

def dispatch(lay: Layout, x_bf16: np.ndarray, q: int, row_begin: int = 0,
             row_end: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Receive rows [row_begin, row_end) as (data bytes [rows, db], scale bytes [rows, sb])."""
    N = lay.R * lay.T
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(N, np.shape(x_bf16)[-1])
    H = x.shape[1]
    if row_end is None:
        row_end = lay.rows
    db, sb = row_bytes(q, H)
    n = row_end - row_begin
    data = np.zeros((n, db), np.uint8)
    scales = np.zeros((n, sb), np.uint8)
    dr = np.ascontiguousarray(lay.dst_row.reshape(-1))
    load().oracle_dispatch(N, lay.K, H, q, _p(dr), _p(x), row_begin, row_end, _p(data),
                           _p(scales) if sb else None)
    return data, scales


def dispatch_scaled(lay: Layout, x_bf16: np.ndarray, q: int, topk: np.ndarray,
                    scales: np.ndarray | None, kind: int, row_begin: int = 0,
                    row_end: int | None = None):
    """Receive rows with input scales of a kind (S_SCALAR [1], S_CHANNEL [H],
    S_EXPERT [E, H]); quantModes 1-3 only."""
    N = lay.R * lay.T
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(N, np.shape(x_bf16)[-1])
    H = x.shape[1]
    if row_end is None:
        row_end = lay.rows
    db, sb = row_bytes(q, H)
    n = row_end - row_begin
    data = np.zeros((n, db), np.uint8)
    scl = np.zeros((n, sb), np.uint8)
    dr = np.ascontiguousarray(lay.dst_row.reshape(-1))
    tk = np.ascontiguousarray(topk, dtype=np.int64).reshape(-1)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    load().oracle_dispatch_scaled(N, lay.K, H, q, _p(dr), _p(tk), _p(x), _p(sc), kind, row_begin,
                                  row_end, _p(data), _p(scl) if sb else None)
    return data, scl


def dispatch_bytes(lay, src_rows: np.ndarray, rows: int | None = None, row_begin: int = 0,
                   out: np.ndarray | None = None) -> np.ndarray:
    """Scatter of already-encoded source rows [N, nbytes] (uint8) onto the
    receive rows [row_begin, rows) of a layout (lay.dst_row, or a TokenLayout's
    tok_dst); rows that no entry reaches are zero.  rows defaults to the
    layout's row count.  out, when given, is a [rows - row_begin, nbytes]
    uint8 buffer to fill (a large receive buffer can be built rank by rank)."""
    N = lay.R * lay.T
    src = np.ascontiguousarray(src_rows, dtype=np.uint8).reshape(N, -1) if N else \
        np.zeros((0, np.shape(src_rows)[-1]), np.uint8)
    nb = src.shape[1]
    dst = lay.tok_dst if hasattr(lay, "tok_dst") else lay.dst_row
    if rows is None:
        rows = lay.rows
    if out is None:
        out = np.zeros((rows - row_begin, nb), np.uint8)
    assert out.shape == (rows - row_begin, nb) and out.dtype == np.uint8 and out.flags.c_contiguous
    dr = np.ascontiguousarray(dst.reshape(-1), dtype=np.int32)
    load().oracle_dispatch_bytes(N, lay.K, _p(dr), _p(src), nb, row_begin, rows, _p(out))
    return out


def return_slots(lay, y_bf16: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Combine send phase of the two-phase form (MAX ep_combine_async): slot
    (s*T + t)*K + k of a token-major buffer holds the expert output row
    dst_row[s,t,k] of y (unweighted).  Returns (slots [R*T*K, H] bf16 bits,
    valid mask [R*T*K]); invalid slots are zero here and unspecified on the
    device."""
    d = np.asarray(lay.dst_row).reshape(-1).astype(np.int64)
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    H = y.shape[-1]
    y = y.reshape(-1, H)
    valid = d >= 0
    out = np.zeros((d.size, H), np.uint16)
    out[valid] = y[d[valid]]
    return out, valid


def slot_layout(lay) -> Layout:
    """The layout the combine wait phase reads: entry (s,t,k) at slot
    (s*T + t)*K + k when valid, -1 otherwise."""
    d = np.asarray(lay.dst_row).reshape(-1)
    ids = np.where(d >= 0, np.arange(d.size), -1).astype(np.int32)
    return Layout(R=lay.R, T=lay.T, K=lay.K, dst_row=ids.reshape(lay.R, lay.T, lay.K))


def transpose_scales(scales_rows: np.ndarray, capacity: int, elem_bytes: int) -> np.ndarray:
    """Row-major receive scales [rows, nb * elem_bytes] (uint8) rearranged into
    the block-major layout of MAX ep_dispatch's output_scales, shape
    (hidden // block_size, max_recv_tokens): element b of row r lands at
    [b, r]; columns past the last row are zero.  Returned as uint8
    [nb, capacity * elem_bytes]."""
    s = np.ascontiguousarray(scales_rows, dtype=np.uint8)
    rows = s.shape[0]
    nb = s.shape[1] // elem_bytes
    out = np.zeros((nb, capacity, elem_bytes), np.uint8)
    out[:, :rows, :] = s.reshape(rows, nb, elem_bytes).transpose(1, 0, 2)
    return out.reshape(nb, capacity * elem_bytes)


def dispatch_rows(lay: Layout, x_bf16: np.ndarray, q: int, rows: np.ndarray):
    """Selected receive rows, computed one by one through recv_src."""
    N = lay.R * lay.T
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(N, np.shape(x_bf16)[-1])
    H = x.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    db, sb = row_bytes(q, H)
    data = np.zeros((len(rows), db), np.uint8)
    scales = np.zeros((len(rows), sb), np.uint8)
    rs = np.ascontiguousarray(lay.recv_src)
    load().oracle_dispatch_rows(len(rows), _p(rows), _p(rs), H, q, _p(x), _p(data),
                                _p(scales) if sb else None)
    return data, scales


def expert_rows(lay: Layout, rows: np.ndarray, H: int, q: int, data: np.ndarray,
                scales: np.ndarray, mark_mod: int = 0) -> np.ndarray:
    """Stand-in expert output (bf16 bits) for receive rows given their bytes."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    re = np.ascontiguousarray(row_expert(lay))
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    y = np.zeros((len(rows), H), np.uint16)
    load().oracle_expert_rows(len(rows), _p(rows), _p(re), H, q, _p(data),
                              _p(scales) if scales.size else None, mark_mod, _p(y))
    return y


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def combine(lay: Layout, y_bf16: np.ndarray, w: np.ndarray, shared: np.ndarray | None = None,
            tok_begin: int = 0, tok_end: int | None = None,
            y_rows: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits of out[tok_begin:tok_end]; y_rows maps receive row -> row of y."""
    R, T, K = lay.R, lay.T, lay.K
    if tok_end is None:
        tok_end = R * T
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    H = y.shape[-1]
    S = 0 if shared is None else shared.shape[1]
    sh = None if shared is None else np.ascontiguousarray(shared, dtype=np.uint16)
    wf = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    dr = np.ascontiguousarray(lay.dst_row.reshape(-1))
    yr = None if y_rows is None else np.ascontiguousarray(y_rows, dtype=np.int64)
    out = np.zeros((tok_end - tok_begin, H), np.uint16)
    load().oracle_combine(R, T, H, K, S, _p(dr), _p(wf), _p(y), _p(yr), _p(sh),
                          tok_begin, tok_end, _p(out))
    return out


def combine_ref64(lay: Layout, y_bf16: np.ndarray, w: np.ndarray,
                  shared: np.ndarray | None = None, tok_begin: int = 0,
                  tok_end: int | None = None, y_rows: np.ndarray | None = None):
    """(fp64 sum, fp64 sum of |terms|) for out[tok_begin:tok_end]."""
    R, T, K = lay.R, lay.T, lay.K
    if tok_end is None:
        tok_end = R * T
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    H = y.shape[-1]
    S = 0 if shared is None else shared.shape[1]
    sh = None if shared is None else np.ascontiguousarray(shared, dtype=np.uint16)
    wf = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    dr = np.ascontiguousarray(lay.dst_row.reshape(-1))
    yr = None if y_rows is None else np.ascontiguousarray(y_rows, dtype=np.int64)
    ref = np.zeros((tok_end - tok_begin, H), np.float64)
    mag = np.zeros((tok_end - tok_begin, H), np.float64)
    load().oracle_combine_ref64(R, T, H, K, S, _p(dr), _p(wf), _p(y), _p(yr), _p(sh),
                                tok_begin, tok_end, _p(ref), _p(mag))
    return ref, mag


# ---------------------------------------------------------------------------
# tolerance
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (normal range: 2^(floor(log2|v|) - 7))."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, e - 8)
    return np.maximum(ulp, np.ldexp(1.0, -133))


def combine_tolerance_floor(mag: np.ndarray, K: int, S: int) -> np.ndarray:
    """Error floor of a binary32 sum of K weighted terms plus S shared terms:
    each multiply and add rounds once (<= 2^-24 relative), so the accumulated
    error is at most (2K + S + 1) * 2^-24 * sum|terms|."""
    return np.ldexp(mag, -24) * (2 * K + S + 1)


def combine_within_tolerance(got_bits: np.ndarray, ref: np.ndarray, mag: np.ndarray,
                             K: int, S: int = 0):
    """Combine tolerance, derived from the arithmetic (fp32 accumulation, one bf16
    rounding at the end):
      every element: |got - ref| <= 2 ulp_bf16(ref) + (2K+S+1) 2^-24 sum|terms|;
      elements with ref != 0 and |ref| >= 2^-10 sum|terms| (no heavy cancellation):
      max |got - ref| / |ref| <= 1e-2.
    ref is the float64 sum.  Returns (ok, max_abs_excess, max_rel)."""
    got = bf16_bits_to_f64(got_bits)
    err = np.abs(got - ref)
    bound = 2.0 * ulp_bf16(ref) + combine_tolerance_floor(mag, K, S)
    excess = float(np.max(err - bound)) if err.size else 0.0
    sel = (np.abs(ref) >= np.ldexp(mag, -10)) & (ref != 0)
    rel = float(np.max(err[sel] / np.abs(ref[sel]))) if np.any(sel) else 0.0
    return bool(excess <= 0.0 and rel <= 1e-2), excess, rel


# ---------------------------------------------------------------------------
# per-rank receive layout (DeepEP recv_x / recv_topk_idx / recv_topk_weights)
# ---------------------------------------------------------------------------

class TokenLayout:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def token_layout(R: int, T: int, E: int, K: int, topk: np.ndarray, w: np.ndarray,
                 mask: np.ndarray | None = None) -> TokenLayout:
    """One receive row per (token, destination rank); a masked entry (xActiveMask)
    takes no part, like a -1 id."""
    N = R * T
    tk = np.ascontiguousarray(topk, dtype=np.int64).reshape(N, K).copy()
    if mask is not None:
        m = np.asarray(mask, np.uint8)
        act = np.repeat(m.reshape(N, 1), K, 1) if m.size == N else m.reshape(N, K)
        tk[act == 0] = -1
    wf = np.ascontiguousarray(w, dtype=np.float32).reshape(N * K)
    cap = max(N * min(R, K), 1)
    tok_dst = np.zeros((N, K), np.int32)
    src = np.zeros(cap, np.int32)
    base = np.zeros(R + 1, np.int64)
    ridx = np.zeros((cap, K), np.int64)
    rw = np.zeros((cap, K), np.float32)
    rows = load().oracle_token_layout(R, T, E, K, _p(tk), _p(wf), cap, _p(tok_dst), _p(src), _p(base),
                                      _p(ridx), _p(rw))
    return TokenLayout(R=R, T=T, E=E, K=K, L=E // R, rows=int(rows), tok_dst=tok_dst,
                       recv_src=src[:rows], rank_tok_base=base, recv_topk_idx=ridx[:rows],
                       recv_topk_weights=rw[:rows])


def token_dispatch(tl: TokenLayout, x_bf16: np.ndarray, q: int):
    """Receive rows of the per-rank layout (the same scatter, onto tok_dst)."""
    N = tl.R * tl.T
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(N, np.shape(x_bf16)[-1])
    H = x.shape[1]
    db, sb = row_bytes(q, H)
    data = np.zeros((tl.rows, db), np.uint8)
    scales = np.zeros((tl.rows, sb), np.uint8)
    dr = np.ascontiguousarray(tl.tok_dst.reshape(-1))
    load().oracle_dispatch(N, tl.K, H, q, _p(dr), _p(x), 0, tl.rows, _p(data), _p(scales) if sb else None)
    return data, scales


def expert_token_rows(tl: TokenLayout, H: int, q: int, data: np.ndarray, scales: np.ndarray,
                      mark_mod: int = 0) -> np.ndarray:
    rows = np.arange(tl.rows, dtype=np.int64)
    y = np.zeros((tl.rows, H), np.uint16)
    d = np.ascontiguousarray(data, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    ridx = np.ascontiguousarray(tl.recv_topk_idx)
    rw = np.ascontiguousarray(tl.recv_topk_weights)
    load().oracle_expert_token_rows(tl.rows, _p(rows), H, tl.K, q, _p(d), _p(sc) if sc.size else None,
                                    _p(ridx), _p(rw), mark_mod, _p(y))
    return y


def token_combine(tl: TokenLayout, y_bf16: np.ndarray, shared: np.ndarray | None = None):
    """out = bf16(sum of the token's per-rank rows + shared rows), unit weights."""
    ones = np.ones((tl.R, tl.T, tl.K), np.float32)
    lay = Layout(R=tl.R, T=tl.T, K=tl.K, dst_row=tl.tok_dst)
    return combine(lay, y_bf16, ones, shared)


def token_combine_ref64(tl: TokenLayout, y_bf16: np.ndarray, shared: np.ndarray | None = None):
    ones = np.ones((tl.R, tl.T, tl.K), np.float32)
    lay = Layout(R=tl.R, T=tl.T, K=tl.K, dst_row=tl.tok_dst)
    return combine_ref64(lay, y_bf16, ones, shared)


def reduce_token_weights(tl: TokenLayout, rank_w: np.ndarray) -> np.ndarray:
    N = tl.R * tl.T
    out = np.zeros((N, tl.K), np.float32)
    rw = np.ascontiguousarray(rank_w, dtype=np.float32)
    load().oracle_reduce_token_weights(N, tl.K, _p(np.ascontiguousarray(tl.tok_dst)), _p(rw), _p(out))
    return out


# ---------------------------------------------------------------------------
# combine + residual add + RMSNorm (CANN aclnnMoeDistributeCombineAddRmsNorm)
# ---------------------------------------------------------------------------

def add_rms_norm_ref64(c: np.ndarray, residual_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float):
    """(x, rstd, y) in float64: x = c + residual, rstd = 1/sqrt(mean(x^2) + eps),
    y = x * rstd * gamma, per row of c [N, H] (float64)."""
    c = np.ascontiguousarray(c, dtype=np.float64)
    N, H = c.shape
    r = np.ascontiguousarray(residual_bf16, dtype=np.uint16).reshape(N, H)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16).reshape(H)
    x = np.zeros((N, H), np.float64)
    rstd = np.zeros(N, np.float64)
    y = np.zeros((N, H), np.float64)
    load().oracle_add_rms_norm_ref64(N, H, _p(c), _p(r), _p(g), float(eps), _p(x), _p(rstd), _p(y))
    return x, rstd, y


def add_rms_norm_f32(c_bf16: np.ndarray, residual_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float):
    """(x bf16 bits, rstd float32, y bf16 bits) of the AddRmsNorm taken step by
    step in binary32 from the combine's bf16 output c [N, H]: x = fl32(c + r),
    a left-to-right binary32 sum of squares, rstd = 1/sqrt(sum/H + eps),
    y = bf16((x * rstd) * gamma)."""
    c = np.ascontiguousarray(c_bf16, dtype=np.uint16)
    N, H = c.shape
    r = np.ascontiguousarray(residual_bf16, dtype=np.uint16).reshape(N, H)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16).reshape(H)
    x = np.zeros((N, H), np.uint16)
    rstd = np.zeros(N, np.float32)
    y = np.zeros((N, H), np.uint16)
    load().oracle_add_rms_norm_f32(N, H, _p(c), _p(r), _p(g), float(eps), _p(x), _p(rstd), _p(y))
    return x, rstd, y


def combine_add_rms_norm_ref64(lay: Layout, y_bf16: np.ndarray, w: np.ndarray, shared, residual_bf16,
                               gamma_bf16, eps: float, tok_begin: int = 0, tok_end: int | None = None,
                               y_rows: np.ndarray | None = None):
    """Reference of the fused combine + AddRmsNorm for tokens [tok_begin, tok_end):
    dict with the exact combine sums c and their magnitudes mag, and x, rstd, y."""
    c, mag = combine_ref64(lay, y_bf16, w, shared, tok_begin, tok_end, y_rows)
    H = c.shape[1]
    r = np.ascontiguousarray(residual_bf16, dtype=np.uint16).reshape(-1, H)
    if r.shape[0] != c.shape[0]:
        r = r[tok_begin:tok_begin + c.shape[0]]
    x, rstd, yv = add_rms_norm_ref64(c, r, gamma_bf16, eps)
    return dict(c=c, mag=mag, x=x, rstd=rstd, y=yv, gamma=bf16_bits_to_f64(gamma_bf16).reshape(H))


def add_rms_norm_within_tolerance(x_bits, rstd, y_bits, ref: dict, K: int, S: int):
    """Derived error bound of a binary32 implementation that rounds the combine
    to bf16 (|c_bf16 - c| <= t = 2 ulp_bf16(c) + (2K+S+1) 2^-24 mag, as for the
    combine), adds the residual in binary32, and normalises in binary32:
      x error   e_i  = t_i + 2^-24 (|x_i| + t_i)
      sum of squares relative error  s = 2 |e|/|x| + (|e|/|x|)^2 + (H+4) 2^-24
      rstd relative error  rho = s / (2 (1 - s)) + 3 * 2^-24
      y error   d_i = |gamma_i| rstd (e_i (1 + rho) + |x_i| rho), plus the
                two binary32 products (2^-22 |y_i|) and the bf16 rounding
                (ulp_bf16 of |y_i| + d_i, twice the half-ulp).
    x_out is checked against e_i + ulp_bf16(|x_i| + e_i).  Returns (ok, worst
    ratio of error to bound over x, rstd, y)."""
    c, mag, x, r, y, g = ref["c"], ref["mag"], ref["x"], ref["rstd"], ref["y"], ref["gamma"]
    H = c.shape[1]
    t = 2.0 * ulp_bf16(c) + (2 * K + S + 1) * 2.0 ** -24 * mag
    e = t + 2.0 ** -24 * (np.abs(x) + t)
    en = np.sqrt((e * e).sum(axis=1))
    xn = np.sqrt((x * x).sum(axis=1))
    q = en / np.maximum(xn, 1e-300)
    s = 2.0 * q + q * q + (H + 4) * 2.0 ** -24
    assert np.all(s < 0.5), "x too small for a meaningful bound"
    rho = s / (2.0 * (1.0 - s)) + 3 * 2.0 ** -24
    out = {}
    gx = bf16_bits_to_f64(np.asarray(x_bits).reshape(x.shape))
    bx = e + ulp_bf16(np.abs(x) + e)
    out["x"] = float(np.max(np.abs(gx - x) / bx)) if x.size else 0.0
    out["rstd"] = float(np.max(np.abs(np.asarray(rstd, np.float64) - r) / (r * rho))) if r.size else 0.0
    d = np.abs(g)[None, :] * r[:, None] * (e * (1.0 + rho[:, None]) + np.abs(x) * rho[:, None])
    by = d * (1.0 + 2.0 ** -20) + 2.0 ** -22 * np.abs(y) + ulp_bf16(np.abs(y) + d)
    gy = bf16_bits_to_f64(np.asarray(y_bits).reshape(y.shape))
    out["y"] = float(np.max(np.abs(gy - y) / by)) if y.size else 0.0
    return all(v <= 1.0 for v in out.values()), out
