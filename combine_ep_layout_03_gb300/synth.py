"""Seeded synthetic inputs for the expert-parallel layout / dispatch / combine path.

This module only draws inputs.  It holds none of the method's arithmetic and
is the one piece of code that both the CUDA path's tests and the CPU oracle's
tests use.  The five workloads are the ones the method is measured on:

  1. R=4 ranks x 64 tokens, H=1024, 16 experts, top-2 distinct uniform, alpha=1
  2. R=8 x 4096, H=7168, 256 experts, top-8 distinct uniform, alpha=1
  3. R=16 x 4096, H=7168 with 1% of rows scaled x100, 256 experts, top-8 drawn
     without replacement from Zipf(s=1.2), per-token int8, alpha=128
  4. R=8 x 8192, H=4096, 128 experts, top-8 uniform, MXFP8 e4m3 then MXFP4 e2m1,
     alpha=128
  5. R=32 x 8192, H=4096, 512 experts, top-16 with 10% of entries set to -1,
     4 shared-expert rows per token added in combine, alpha=64

Recipe (seed = 1000 + workload index, numpy PCG64 unless noted):
  - routing "uniform": per token, the K smallest of E uniform keys, slots in
    ascending key order (a uniformly random ordered K-subset);
  - routing "zipf": p(e) ~ (e+1)^-s over e in [0, E) (no permutation, so the hot
    experts sit on rank 0), K distinct by Gumbel-top-K: keys = log p(e) + Gumbel,
    slots in descending key order;
  - drop: each entry set to -1 independently with probability drop_p, after
    drawing;
  - weights: logits N(0,1), softmax in float64 over the valid entries of the
    token, cast to float32; invalid entries get weight 0;
  - x: float32 N(0,1), outlier rows (Bernoulli(outlier_p) per token) multiplied
    by outlier_scale, then rounded once to bf16 (torch's round-to-nearest-even
    cast).  For the full-size workloads x and the shared-expert rows can be drawn
    on the GPU instead (torch Philox generator, same seed), because drawing
    billions of normals on the host takes minutes.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

QUANT_NAMES = {0: "none", 1: "int8_static", 2: "int8", 4: "mxfp8_e4m3", 5: "mxfp8_e5m2", 6: "mxfp4_e2m1",
               7: "fp8_e4m3_token", 8: "fp8_e5m2_token", 9: "fp8_e4m3_group128", 10: "fp8_e5m2_group128"}


@dataclass(frozen=True)
class Workload:
    index: int
    R: int
    T: int
    H: int
    E: int
    K: int
    alpha: int
    quants: tuple = (0,)
    routing: str = "uniform"
    zipf_s: float = 1.2
    drop_p: float = 0.0
    outlier_p: float = 0.0
    outlier_scale: float = 100.0
    num_shared: int = 0

    @property
    def N(self) -> int:
        return self.R * self.T

    @property
    def L(self) -> int:
        return self.E // self.R

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def name(self) -> str:
        q = "+".join(QUANT_NAMES[m] for m in self.quants)
        return (f"R{self.R}_T{self.T}_H{self.H}_E{self.E}_K{self.K}_a{self.alpha}"
                f"_{self.routing}{'_drop' + str(self.drop_p) if self.drop_p else ''}"
                f"{'_S' + str(self.num_shared) if self.num_shared else ''}_{q}")

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    1: Workload(1, R=4, T=64, H=1024, E=16, K=2, alpha=1),
    2: Workload(2, R=8, T=4096, H=7168, E=256, K=8, alpha=1),
    3: Workload(3, R=16, T=4096, H=7168, E=256, K=8, alpha=128, quants=(2,),
                routing="zipf", zipf_s=1.2, outlier_p=0.01, outlier_scale=100.0),
    4: Workload(4, R=8, T=8192, H=4096, E=128, K=8, alpha=128, quants=(4, 6)),
    5: Workload(5, R=32, T=8192, H=4096, E=512, K=16, alpha=64, drop_p=0.1, num_shared=4),
}


def _rng(w: Workload, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, stream]))


def gen_topk(w: Workload, chunk: int = 16384) -> np.ndarray:
    """topk_idx [R, T, K] int64."""
    rng = _rng(w, 0)
    N, E, K = w.N, w.E, w.K
    out = np.empty((N, K), np.int64)
    if w.routing == "uniform":
        for a in range(0, N, chunk):
            b = min(N, a + chunk)
            keys = rng.random((b - a, E))
            part = np.argpartition(keys, K - 1, axis=1)[:, :K]
            pk = np.take_along_axis(keys, part, axis=1)
            order = np.argsort(pk, axis=1, kind="stable")
            out[a:b] = np.take_along_axis(part, order, axis=1)
    elif w.routing == "zipf":
        logp = -w.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        for a in range(0, N, chunk):
            b = min(N, a + chunk)
            keys = logp[None, :] + rng.gumbel(size=(b - a, E))
            part = np.argpartition(-keys, K - 1, axis=1)[:, :K]
            pk = np.take_along_axis(keys, part, axis=1)
            order = np.argsort(-pk, axis=1, kind="stable")
            out[a:b] = np.take_along_axis(part, order, axis=1)
    else:
        raise ValueError(w.routing)
    if w.drop_p > 0:
        drop = _rng(w, 1).random((N, K)) < w.drop_p
        out[drop] = -1
    return out.reshape(w.R, w.T, K)


def gen_weights(w: Workload, topk: np.ndarray) -> np.ndarray:
    """topk_weights [R, T, K] float32: softmax over each token's valid entries."""
    rng = _rng(w, 2)
    tk = topk.reshape(w.N, w.K)
    logits = rng.standard_normal((w.N, w.K))
    valid = tk >= 0
    z = np.where(valid, logits, -np.inf)
    m = np.max(z, axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    ex = np.where(valid, np.exp(z - m), 0.0)
    den = ex.sum(axis=1, keepdims=True)
    wts = np.where(den > 0, ex / np.where(den > 0, den, 1.0), 0.0)
    return wts.astype(np.float32).reshape(w.R, w.T, w.K)


def _to_bf16_bits(xf32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(xf32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def gen_x(w: Workload, chunk: int = 1 << 24) -> np.ndarray:
    """x [R, T, H] as bf16 bit patterns (uint16), drawn on the host."""
    rng = _rng(w, 3)
    N, H = w.N, w.H
    out = np.empty((N, H), np.uint16)
    rows = max(1, chunk // H)
    outl = _rng(w, 4).random(N) < w.outlier_p if w.outlier_p > 0 else None
    for a in range(0, N, rows):
        b = min(N, a + rows)
        xf = rng.standard_normal((b - a, H), dtype=np.float32)
        if outl is not None:
            xf[outl[a:b]] *= np.float32(w.outlier_scale)
        out[a:b] = _to_bf16_bits(xf)
    return out.reshape(w.R, w.T, H)


def gen_shared(w: Workload, chunk: int = 1 << 24) -> np.ndarray | None:
    """Shared-expert outputs [R, S, T, H] bf16 bits, or None when S = 0."""
    if w.num_shared == 0:
        return None
    rng = _rng(w, 5)
    total = w.R * w.num_shared * w.T
    out = np.empty((total, w.H), np.uint16)
    rows = max(1, chunk // w.H)
    for a in range(0, total, rows):
        b = min(total, a + rows)
        out[a:b] = _to_bf16_bits(rng.standard_normal((b - a, w.H), dtype=np.float32))
    return out.reshape(w.R, w.num_shared, w.T, w.H)


def gen_y(w: Workload, rows: int, stream: int = 6) -> np.ndarray:
    """Independent bf16 expert outputs [rows, H] (bits), for combine-only tests."""
    rng = _rng(w, stream)
    return _to_bf16_bits(rng.standard_normal((rows, w.H), dtype=np.float32))


def gen_x_device(w: Workload, device="cuda") -> torch.Tensor:
    """x [R, T, H] bf16 drawn on the GPU (torch Philox, seeded), same recipe."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    x = torch.randn((w.N, w.H), generator=g, device=device, dtype=torch.float32)
    if w.outlier_p > 0:
        outl = torch.rand((w.N,), generator=g, device=device) < w.outlier_p
        x[outl] *= w.outlier_scale
    return x.to(torch.bfloat16).view(w.R, w.T, w.H)


def gen_shared_device(w: Workload, device="cuda") -> torch.Tensor | None:
    if w.num_shared == 0:
        return None
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 7919)
    out = torch.empty((w.R, w.num_shared, w.T, w.H), device=device, dtype=torch.bfloat16)
    flat = out.view(-1, w.H)
    step = max(1, (1 << 26) // w.H)
    for a in range(0, flat.shape[0], step):
        b = min(flat.shape[0], a + step)
        flat[a:b] = torch.randn((b - a, w.H), generator=g, device=device).to(torch.bfloat16)
    return out


def gen_scales(w: Workload, kind: int, stream: int = 7) -> np.ndarray | None:
    """Input scales of quantModes 1-3: kind 1 -> [1], 2 -> [H], 3 -> [E, H];
    float32 uniform in [0.5, 2) (a smooth weight around 1).  kind 0 -> None."""
    if kind == 0:
        return None
    rng = _rng(w, stream)
    shape = {1: (1,), 2: (w.H,), 3: (w.E, w.H)}[kind]
    return (0.5 + 1.5 * rng.random(shape)).astype(np.float32)


def gen_mask(w: Workload, dims: int, p_active: float = 0.9, stream: int = 8) -> np.ndarray:
    """xActiveMask: uint8 [R, T] (dims 1) or [R, T, K] (dims 2), Bernoulli(p_active)."""
    rng = _rng(w, stream)
    shape = (w.R, w.T) if dims == 1 else (w.R, w.T, w.K)
    return (rng.random(shape) < p_active).astype(np.uint8)


def gen_encoded_rows(w: Workload, data_bytes: int, scale_bytes: int, stream: int = 9):
    """Already-encoded source rows for the pre-encoded dispatch: uint8 data
    [N, data_bytes] and scales [N, scale_bytes], every byte uniform in [0, 256).
    The dispatch moves these bytes without reading them as numbers, so any
    byte pattern is a valid input."""
    rng = _rng(w, stream)
    data = rng.integers(0, 256, size=(w.N, data_bytes), dtype=np.uint8)
    scales = rng.integers(0, 256, size=(w.N, scale_bytes), dtype=np.uint8)
    return data, scales


def gen_encoded_rows_device(w: Workload, data_bytes: int, scale_bytes: int, device="cuda"):
    """gen_encoded_rows drawn on the GPU (torch Philox, seeded) for full sizes."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 4099)
    data = torch.randint(0, 256, (w.N, data_bytes), generator=g, device=device, dtype=torch.uint8)
    scales = torch.randint(0, 256, (w.N, scale_bytes), generator=g, device=device, dtype=torch.uint8)
    return data, scales


RMS_NORM_EPS = 1e-6


def gen_residual(w: Workload, stream: int = 10, chunk: int = 1 << 24) -> np.ndarray:
    """Residual rows of the combine + AddRmsNorm step, [R, T, H] bf16 bits:
    float32 N(0,1) rounded once to bf16."""
    rng = _rng(w, stream)
    out = np.empty((w.N, w.H), np.uint16)
    rows = max(1, chunk // w.H)
    for a in range(0, w.N, rows):
        b = min(w.N, a + rows)
        out[a:b] = _to_bf16_bits(rng.standard_normal((b - a, w.H), dtype=np.float32))
    return out.reshape(w.R, w.T, w.H)


def gen_gamma(w: Workload, stream: int = 11) -> np.ndarray:
    """RMSNorm weight gamma [H] bf16 bits: 1 + 0.1 * N(0,1), rounded to bf16."""
    rng = _rng(w, stream)
    return _to_bf16_bits((1.0 + 0.1 * rng.standard_normal(w.H)).astype(np.float32))


def gen_residual_device(w: Workload, device="cuda") -> torch.Tensor:
    """gen_residual's recipe drawn on the GPU (torch Philox, seeded) for full sizes."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 6007)
    return torch.randn((w.N, w.H), generator=g, device=device).to(torch.bfloat16).view(w.R, w.T, w.H)
