"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/ep_layout.h declares, and rejects invalid arguments on the host before
any CUDA call (the aclnn convention of validating in the first phase)."""
import ctypes
import os
import re
import subprocess

import pytest

from combine_ep_layout_03_gb300 import ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep_layout.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = set(re.findall(r"\b(ep_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ep_layout", "ep_dispatch", "ep_combine", "ep_layout_workspace_size",
                 "ep_handle_create", "ep_handle_destroy", "ep_handle_status"):
        assert must in names


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", ep.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert getattr(ep.lib, n) is not None


def good():
    return ep.make_params(8, 4096, 7168, 256, 8, 1, 0)


@pytest.mark.parametrize("field,value", [
    ("num_ranks", 0), ("num_experts", 0), ("num_experts", 513), ("num_experts", 250),
    ("topk", 0), ("topk", 17), ("tokens_per_rank", -1), ("tokens_per_rank", 65537),
    ("hidden", 0), ("hidden", 7164), ("hidden", 8200), ("expert_alignment", 0),
    ("recv_capacity_rows", -5)])
def test_validation_rejects(field, value):
    p = good()
    setattr(p, field, value)
    assert ep.ep_params_validate(p) == ep.EP_ERR_INVALID_ARG
    with pytest.raises(ep.EPError) as ei:
        ep.ep_layout_workspace_size(p)
    assert ei.value.status == ep.EP_ERR_INVALID_ARG


def test_topk_larger_than_experts_rejected():
    p = ep.make_params(2, 8, 64, 4, 5, 1, 0)
    assert ep.ep_params_validate(p) == ep.EP_ERR_INVALID_ARG


def test_validation_accepts_the_workloads():
    from combine_ep_layout_03_gb300 import synth
    for w in synth.WORKLOADS.values():
        p = ep.make_params(w.R, w.T, w.H, w.E, w.K, w.alpha, 0)
        assert ep.ep_params_validate(p) == ep.EP_OK
    assert ep.ep_params_validate(ep.make_params(4, 0, 1024, 16, 2, 1, 0)) == ep.EP_OK  # T = 0


def test_row_bytes():
    assert ep.ep_recv_row_bytes(7168, ep.EP_QUANT_NONE) == (14336, 0)
    assert ep.ep_recv_row_bytes(7168, ep.EP_QUANT_INT8_PER_TOKEN) == (7168, 4)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_MXFP8_E4M3) == (4096, 128)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_MXFP8_E5M2) == (4096, 128)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_MXFP4_E2M1) == (2048, 128)
    with pytest.raises(ep.EPError):
        ep.ep_recv_row_bytes(4104, ep.EP_QUANT_MXFP8_E4M3)  # H % 32 != 0 for MX
    with pytest.raises(ep.EPError) as ei:
        ep.ep_recv_row_bytes(4096, 3)
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED


def _create_fake(p, base=1 << 40):
    """Handle over a fake, never dereferenced device address (host-only calls)."""
    n = ep.ep_layout_workspace_size(p)
    h = ctypes.c_void_p(0)
    st = ep.lib.ep_handle_create(ctypes.byref(p), base, n, ctypes.byref(h))
    return st, h.value, n


def test_workspace_carving_is_aligned_and_disjoint():
    from combine_ep_layout_03_gb300.ep import _VIEW_SPECS
    for w in (ep.make_params(8, 4096, 7168, 256, 8, 1, 0), ep.make_params(32, 8192, 4096, 512, 16, 64, 0),
              ep.make_params(3, 0, 64, 6, 2, 4, 0), ep.make_params(2, 5, 16, 2, 2, 3, 100)):
        st, h, n = _create_fake(w)
        assert st == ep.EP_OK
        v = ep.ep_handle_views(h)
        R, T, E, K = w.num_ranks, w.tokens_per_rank, w.num_experts, w.topk

        class S:
            pass
        s = S()
        s.R, s.T, s.E, s.K, s.L = R, T, E, K, E // R
        s.recv_src_capacity = v.recv_src_capacity
        s.tok_capacity = v.tok_capacity
        assert v.tok_capacity == R * T * min(R, K)
        worst = R * T * K + E * (w.expert_alignment - 1)
        assert v.recv_src_capacity == (w.recv_capacity_rows or worst)
        spans = []
        for name, (dt, shape) in _VIEW_SPECS.items():
            ptr = getattr(v, name)
            size = 1
            for d in shape(s):
                size *= d
            nbytes = size * {1: 1, 4: 4, 8: 8}[{"torch.uint8": 1, "torch.int32": 4, "torch.int64": 8}[str(dt)]]
            assert (ptr - (1 << 40)) % 256 == 0, name
            spans.append((ptr, ptr + nbytes, name))
        spans.sort()
        for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
            assert a1 <= b0, (na, nb)
        assert spans[-1][1] <= (1 << 40) + n
        ep.ep_handle_destroy(h)


def test_create_rejects_bad_workspace():
    p = good()
    n = ep.ep_layout_workspace_size(p)
    h = ctypes.c_void_p(0)
    assert ep.lib.ep_handle_create(ctypes.byref(p), (1 << 40) + 8, n, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_handle_create(ctypes.byref(p), 1 << 40, n - 1, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_handle_create(ctypes.byref(p), None, n, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG


def test_launching_calls_validate_before_touching_cuda():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    assert st == ep.EP_OK
    L = ep.lib
    # unsupported quant mode, unaligned pointers, negative capacities
    assert L.ep_dispatch(h, 1 << 40, 3, 1 << 41, None, 10, None) == ep.EP_ERR_UNSUPPORTED
    assert L.ep_dispatch(h, (1 << 40) + 2, 0, 1 << 41, None, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(h, 1 << 40, 2, 1 << 41, None, 10, None) == ep.EP_ERR_INVALID_ARG  # no scales
    assert L.ep_dispatch(h, 1 << 40, 0, 1 << 41, None, -1, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_combine(h, 1 << 40, 10, None, None, 0, 1 << 41, None) == ep.EP_ERR_INVALID_ARG  # no weights
    assert L.ep_combine(h, 1 << 40, 10, 1 << 42, None, 2, 1 << 41, None) == ep.EP_ERR_INVALID_ARG  # no shared
    assert L.ep_combine(h, 1 << 40, 10, 1 << 42, None, 0, (1 << 41) + 4, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_layout(h, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_expert_identity(h, 11, 1 << 40, None, 4, 0, 1 << 41, None) == ep.EP_ERR_UNSUPPORTED
    assert L.ep_expert_identity(h, 0, 1 << 40, None, 4, -1, 1 << 41, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_layout(None, None, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)
    # MX dispatch on a hidden size that is not a multiple of 32
    p = ep.make_params(2, 8, 40, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    assert L.ep_dispatch(h, 1 << 40, 4, 1 << 41, 1 << 42, 10, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)


def test_status_strings():
    for code, name in [(0, "EP_OK"), (1, "EP_ERR_INVALID_ARG"), (3, "EP_ERR_CAPACITY"),
                       (4, "EP_ERR_BAD_EXPERT_ID"), (6, "EP_ERR_CUDA")]:
        assert ep.status_string(code) == name


def test_combine_rejects_too_many_shared_rows():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    assert ep.lib.ep_combine(h, 1 << 40, 10, 1 << 42, 1 << 43, 17, 1 << 41, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)


def test_scaled_dispatch_and_mask_validation():
    p = ep.make_params(2, 8, 256, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C = 1 << 40, 1 << 41, 1 << 42
    # static int8 needs scales; MX and bf16 take none; unknown kind; unaligned per-channel scales
    assert L.ep_dispatch_scaled(h, A, 1, None, 0, B, None, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_scaled(h, A, 4, C, 2, B, C, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_scaled(h, A, 0, C, 1, B, None, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_scaled(h, A, 2, C, 7, B, C, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_scaled(h, A, 2, C + 4, 2, B, C, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_scaled(h, A, 9, None, 0, B, None, 10, None) == ep.EP_ERR_INVALID_ARG  # no scale buffer
    assert L.ep_dispatch_scaled(h, A, 11, None, 0, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED
    # mask dims must be 1 or 2
    assert L.ep_layout_masked(h, A, B, 3, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)
    # per-group FP8 needs H % 128 == 0
    p = ep.make_params(2, 8, 96, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    assert L.ep_dispatch_scaled(h, A, 9, None, 0, B, C, 10, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)


def test_row_bytes_new_modes():
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_INT8_STATIC) == (4096, 0)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_FP8_E4M3_PER_TOKEN) == (4096, 4)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_FP8_E5M2_PER_TOKEN) == (4096, 4)
    assert ep.ep_recv_row_bytes(4096, ep.EP_QUANT_FP8_E4M3_PER_GROUP) == (4096, 128)
    assert ep.ep_recv_row_bytes(7168, ep.EP_QUANT_FP8_E5M2_PER_GROUP) == (7168, 224)
    with pytest.raises(ep.EPError):
        ep.ep_recv_row_bytes(4160, ep.EP_QUANT_FP8_E4M3_PER_GROUP)


def test_token_layout_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C, D = 1 << 40, 1 << 41, 1 << 42, 1 << 43
    assert L.ep_token_layout(h, A, None, None, 0, C, D, 10, None) == ep.EP_ERR_INVALID_ARG   # no weights
    assert L.ep_token_layout(h, A, B, None, 0, None, D, 10, None) == ep.EP_ERR_INVALID_ARG   # no idx out
    assert L.ep_token_layout(h, A, B, C, 5, C, D, 10, None) == ep.EP_ERR_INVALID_ARG        # mask dims
    assert L.ep_dispatch_tokens(h, A, 2, C, 3, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED      # per-expert
    assert L.ep_combine_tokens(h, A, 10, None, 0, B, C, None, None) == ep.EP_ERR_INVALID_ARG  # weights pair
    assert L.ep_expert_identity_tokens(h, 0, A, None, None, B, 4, 0, C, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)


def test_dispatch_ex_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C, D = 1 << 40, 1 << 41, 1 << 42, 1 << 43
    PRE, BM, RANK = ep.EP_DISPATCH_PRE_ENCODED, ep.EP_DISPATCH_SCALES_BLOCK_MAJOR, ep.EP_DISPATCH_PER_RANK
    assert L.ep_dispatch_ex(h, A, None, 4, None, 0, 8, B, C, 10, None) == ep.EP_ERR_INVALID_ARG   # unknown flag
    assert L.ep_dispatch_ex(h, A, None, 4, None, 0, PRE, B, C, 10, None) == ep.EP_ERR_INVALID_ARG  # no x_scales
    assert L.ep_dispatch_ex(h, A, D + 2, 4, None, 0, PRE, B, C, 10, None) == ep.EP_ERR_INVALID_ARG  # unaligned
    assert L.ep_dispatch_ex(h, A, D, 0, None, 0, PRE, B, None, 10, None) == ep.EP_ERR_INVALID_ARG  # bf16 has none
    assert L.ep_dispatch_ex(h, A, D, 2, C, 2, PRE, B, C, 10, None) == ep.EP_ERR_INVALID_ARG  # scales on encoded rows
    assert L.ep_dispatch_ex(h, A, D, 4, None, 0, BM, B, C, 10, None) == ep.EP_ERR_INVALID_ARG  # x_scales w/o PRE
    assert L.ep_dispatch_ex(h, A, None, 2, C, 3, RANK, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED  # per-expert
    assert L.ep_dispatch_ex(h, A, None, 11, None, 0, 0, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED
    ep.ep_handle_destroy(h)
    # encoded int8 rows of H = 72 bytes are not whole 16-byte units: no bulk copy
    p = ep.make_params(2, 8, 72, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    assert L.ep_dispatch_ex(h, A, D, 2, None, 0, PRE, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED
    ep.ep_handle_destroy(h)


def test_combine_add_rms_norm_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C, D, E_ = 1 << 40, 1 << 41, 1 << 42, 1 << 43, 1 << 44
    nan = float("nan")
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, None, D, 1e-6, E_, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # no residual
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, None, 1e-6, E_, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # no gamma
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, D + 8, 1e-6, E_, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # unaligned gamma
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, D, -1.0, E_, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # negative eps
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, D, nan, E_, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # NaN eps
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, D, 1e-6, None, None, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # no output
    assert L.ep_combine_add_rms_norm(h, A, 10, B, None, 0, C, D, 1e-6, E_, E_ + 2, None, None) \
        == ep.EP_ERR_INVALID_ARG                                                            # unaligned x_out
    ep.ep_handle_destroy(h)


def test_two_phase_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C, D = 1 << 40, 1 << 41, 1 << 42, 1 << 43
    NK = 2 * 8 * 2
    assert L.ep_dispatch_async(h, A, 2, C, 3, B, C, 10, None) == ep.EP_ERR_UNSUPPORTED       # per-expert
    assert L.ep_dispatch_wait(h, 4, A, B, 10, 1, C, D, 10, None) == ep.EP_ERR_INVALID_ARG    # per-rank flag
    assert L.ep_dispatch_wait(h, 4, A, None, 10, 0, C, D, 10, None) == ep.EP_ERR_INVALID_ARG  # no arrival scales
    assert L.ep_dispatch_wait(h, 0, A + 8, None, 10, 0, C, None, 10, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_wait(h, 11, A, None, 10, 0, C, None, 10, None) == ep.EP_ERR_UNSUPPORTED
    assert L.ep_combine_async(h, A, 10, B, NK - 1, None) == ep.EP_ERR_INVALID_ARG           # return too small
    assert L.ep_combine_async(h, A, 10, B + 4, NK, None) == ep.EP_ERR_INVALID_ARG           # unaligned
    assert L.ep_combine_wait(h, A, NK - 1, B, None, 0, C, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_combine_wait(h, A, NK, None, None, 0, C, None) == ep.EP_ERR_INVALID_ARG     # no weights
    ep.ep_handle_destroy(h)


def test_stalled_combine_hook_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C = 1 << 40, 1 << 41, 1 << 42
    assert L.ep_test_combine_stalled(h, A, 10, B, C, 0, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_test_combine_stalled(h, A, 10, B, C, (1 << 22) + 1, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_test_combine_stalled(h, A, 10, None, C, 16, None) == ep.EP_ERR_INVALID_ARG
    ep.ep_handle_destroy(h)


def test_step_host_validation():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    st, h, _ = _create_fake(p)
    L = ep.lib
    A, B, C, D = 1 << 40, 1 << 41, 1 << 42, 1 << 43
    bufs = ep.ep_step_buffers()
    bufs.topk, bufs.weights, bufs.x, bufs.out, bufs.recv_data = A, B, C, D, A
    bufs.recv_rows_capacity = 64
    ref = ctypes.byref(bufs)
    assert L.ep_step_host(h, 0, A, B, C, None, 0, D, None, None) == ep.EP_ERR_INVALID_ARG      # no buffers
    assert L.ep_step_host(h, 4, A, B, C, None, 0, D, ref, None) == ep.EP_ERR_INVALID_ARG       # quantised, no y
    assert L.ep_step_host(h, 0, A, B, C, None, 17, D, ref, None) == ep.EP_ERR_INVALID_ARG      # too many shared
    assert L.ep_step_host(h, 0, A, B, C, None, 2, D, ref, None) == ep.EP_ERR_INVALID_ARG       # shared missing
    assert L.ep_step_host(h, 0, None, B, C, None, 0, D, ref, None) == ep.EP_ERR_INVALID_ARG    # no host topk
    assert L.ep_step_host(h, 11, A, B, C, None, 0, D, ref, None) == ep.EP_ERR_UNSUPPORTED
    ep.ep_handle_destroy(h)


def test_static_scratch_layout_refuses_misaligned_pointers_before_any_launch():
    p = ep.make_params(2, 8, 64, 4, 2, 1, 0)
    L = ep.lib
    names = [n for n, _ in ep.ep_layout_outputs._fields_]

    def outputs(**override):
        vals = {n: (1 << 40) + (i << 20) for i, n in enumerate(names)}   # aligned stand-ins
        vals.update(override)
        return ctypes.byref(ep.ep_layout_outputs(**vals))

    topk_ok = 1 << 44
    # topk_idx is read as int64 words
    for off in (1, 4):
        assert L.ep_layout_static_scratch(p, topk_ok + off, outputs(), None) == ep.EP_ERR_INVALID_ARG
    # int32 outputs need 4-byte and rank_base 8-byte alignment
    assert L.ep_layout_static_scratch(p, topk_ok, outputs(dst_row=(1 << 40) + 2), None) == \
        ep.EP_ERR_INVALID_ARG
    assert L.ep_layout_static_scratch(p, topk_ok, outputs(rank_base=(1 << 40) + 4), None) == \
        ep.EP_ERR_INVALID_ARG
    assert L.ep_layout_static_scratch(p, topk_ok, outputs(status=None), None) == ep.EP_ERR_INVALID_ARG
