"""Seeded synthetic inputs for the ZeRO update step.

This module holds no arithmetic of the step itself: it only draws random
gradients, master weights and tensor-size lists with fixed seeds, so that the
CUDA path and the CPU oracle can be fed the very same inputs.  Everything is
generated with torch's generators (on the CPU for small cases, on the GPU for
full-size workloads) and handed to both sides as plain buffers.

Workloads (sizes as the benchmark and the parity tests use them):

* ``flat1m_n4``: flat vector of 1,048,576 parameters, N=4 ranks, BF16 grads
  ~N(0, 1e-3), master ~N(0, 0.02), Adam lr 1e-3, 3 steps.
* ``gpt2small_n4``: the GPT-2-small tensor list (123,588,864 parameters,
  padded to 123,589,120), N=4, BF16 grads ~N(0, 1e-3), AdamW wd 0.1, 10 steps.
* ``flat1b_n8``: 1,000,000,000 parameters, N=8, BF16 grads ~N(0, 5e-4) held
  loss-scaled, 25,000,000-element buckets, dynamic loss scale from 65536, one
  +inf injected on step 3 (that step must be skipped), 5 steps.
* ``flat3b_n4_fp32``: 3,000,000,000 parameters, N=4, FP32 grads ~N(0, 1e-3),
  global-norm clip at 1.0, 3 steps.
* ``ragged6b_n4``: 6,000,000,007 parameters in tensors of mixed sizes 1..2^27
  (the last shard ragged and padded), N=4, BF16 grads ~N(0, 1e-3) with 0.1%
  outliers ~N(0, 1), Adam lr 3e-4, 2 steps.

No public dataset or trained weights are involved: GPT-2-small contributes
only its tensor shapes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 0x5EED0000
GPT2_SMALL_D = 768
GPT2_SMALL_VOCAB = 50257
GPT2_SMALL_LAYERS = 12


def gpt2_small_tensor_sizes() -> list[int]:
    """Element counts of the GPT-2-small tensors: token embedding 50257x768,
    then per layer ln1 weight/bias, qkv 768x2304, attention projection
    768x768 and its bias, ln2 weight/bias, MLP 768x3072 and 3072x768 and the
    MLP projection bias; then the final layer-norm weight and bias."""
    d = GPT2_SMALL_D
    sizes = [GPT2_SMALL_VOCAB * d]
    for _ in range(GPT2_SMALL_LAYERS):
        sizes += [d, d, d * 3 * d, d * d, d, d, d, d * 4 * d, 4 * d * d, d]
    sizes += [d, d]
    return sizes


def mixed_tensor_sizes(total: int, seed: int, lo: int = 1, hi: int = 1 << 27) -> list[int]:
    """Seeded log-uniform tensor sizes in [lo, hi] (both ends included once),
    concatenated until they sum to exactly ``total``; the last is trimmed."""
    rng = np.random.Generator(np.random.Philox(seed))
    sizes = [lo, hi]
    acc = lo + hi
    while acc < total:
        s = int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        s = max(lo, min(hi, s))
        s = min(s, total - acc)
        sizes.append(s)
        acc += s
    assert acc == total
    return sizes


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    grad_dtype: str               # "bf16" | "fp32"
    sigma: float                  # std of the batch-mean per-rank gradient
    steps: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_grad_norm: float = 0.0
    loss_scale: float = 1.0
    dynamic_loss_scale: bool = False
    skip_on_overflow: bool = False
    bucket_elems: int = 0
    inject_inf_step: int = 0      # 1-based step that gets one +inf, 0 = none
    outlier_frac: float = 0.0
    outlier_sigma: float = 1.0
    master_sigma: float = 0.02
    tensor_sizes: tuple = field(default=(), repr=False)
    psi_flat: int = 0             # used when tensor_sizes is empty
    index: int = 0                # seed namespace

    @property
    def sizes(self) -> list[int]:
        return list(self.tensor_sizes) if self.tensor_sizes else [self.psi_flat]

    @property
    def psi(self) -> int:
        return int(sum(self.sizes))

    @property
    def psi_pad(self) -> int:
        unit = self.N * 128
        return -(-self.psi // unit) * unit

    @property
    def grad_bytes(self) -> int:
        return 2 if self.grad_dtype == "bf16" else 4


def _wl(**kw) -> Workload:
    return Workload(**kw)


WORKLOADS: dict[str, Workload] = {
    "flat1m_n4": _wl(name="flat1m_n4", index=1, N=4, grad_dtype="bf16", sigma=1e-3,
                     steps=3, psi_flat=1_048_576),
    "gpt2small_n4": _wl(name="gpt2small_n4", index=2, N=4, grad_dtype="bf16", sigma=1e-3,
                        steps=10, weight_decay=0.1,
                        tensor_sizes=tuple(gpt2_small_tensor_sizes())),
    "flat1b_n8": _wl(name="flat1b_n8", index=3, N=8, grad_dtype="bf16", sigma=5e-4, steps=5,
                     loss_scale=65536.0, dynamic_loss_scale=True, skip_on_overflow=True,
                     bucket_elems=25_000_000, inject_inf_step=3, psi_flat=1_000_000_000),
    "flat3b_n4_fp32": _wl(name="flat3b_n4_fp32", index=4, N=4, grad_dtype="fp32", sigma=1e-3,
                          steps=3, max_grad_norm=1.0, psi_flat=3_000_000_000),
    "ragged6b_n4": _wl(name="ragged6b_n4", index=5, N=4, grad_dtype="bf16", sigma=1e-3,
                       steps=2, lr=3e-4, outlier_frac=1e-3, outlier_sigma=1.0,
                       psi_flat=6_000_000_007),
}


def ragged6b_tensor_sizes() -> list[int]:
    """The mixed per-tensor sizes of ``ragged6b_n4`` (about 90 tensors)."""
    return mixed_tensor_sizes(6_000_000_007, seed=SEED_BASE + 500)


def seed_for(wl_index: int, step: int, rank: int) -> int:
    """Seed of rank ``rank``'s gradient on 1-based ``step``; rank 9 of step 0
    is reserved for the master weights."""
    return SEED_BASE + 100 * wl_index + 10 * step + rank


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_CHUNK = 1 << 26


def fill_normal_(out: torch.Tensor, n_valid: int, sigma: float, seed: int,
                 outlier_frac: float = 0.0, outlier_sigma: float = 1.0) -> torch.Tensor:
    """Fill the flat tensor ``out`` (bf16 or fp32) with sigma * N(0, 1) draws
    on [0, n_valid) and zeros on the padding, chunk by chunk.  With
    ``outlier_frac`` > 0 each element is independently replaced, with that
    probability, by an outlier_sigma * N(0, 1) draw.  BF16 outputs are the
    round-to-nearest-even cast of the FP32 draws (torch's own cast)."""
    gen = _gen(seed, out.device)
    flat = out.view(-1)
    for start in range(0, n_valid, _CHUNK):
        n = min(_CHUNK, n_valid - start)
        z = torch.randn(n, generator=gen, device=out.device, dtype=torch.float32)
        z.mul_(sigma)
        if outlier_frac > 0.0:
            u = torch.rand(n, generator=gen, device=out.device, dtype=torch.float32)
            big = torch.randn(n, generator=gen, device=out.device, dtype=torch.float32)
            big.mul_(outlier_sigma)
            z = torch.where(u < outlier_frac, big, z)
        flat[start:start + n].copy_(z)
        del z
    if flat.numel() > n_valid:
        flat[n_valid:].zero_()
    return out


def inf_index(wl: Workload, step: int) -> tuple[int, int]:
    """(rank, flat index) that receives the injected +inf on ``step``."""
    rng = np.random.Generator(np.random.Philox(seed_for(wl.index, step, 8)))
    return 1 % wl.N, int(rng.integers(0, wl.psi))


def torch_grad_dtype(wl: Workload) -> torch.dtype:
    return torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32


def make_grads(wl: Workload, step: int, device, loss_scale: float | None = None,
               out: list[torch.Tensor] | None = None, psi_pad: int | None = None,
               psi: int | None = None) -> list[torch.Tensor]:
    """The N ranks' gradient buffers for 1-based ``step``.

    Each rank's buffer holds its contribution to the loss-scaled gradient,
    loss_scale * sigma * z with z ~ N(0, 1) drawn independently per rank, so
    after the step divides the sum by N * loss_scale the combined gradient has
    per-element std sigma / sqrt(N).  ``psi``/``psi_pad`` override the
    workload's sizes (for reduced cases)."""
    psi = wl.psi if psi is None else psi
    psi_pad = wl.psi_pad if psi_pad is None else psi_pad
    scale = wl.loss_scale if loss_scale is None else loss_scale
    dt = torch_grad_dtype(wl)
    if out is None:
        out = [torch.empty(psi_pad, dtype=dt, device=device) for _ in range(wl.N)]
    for r in range(wl.N):
        fill_normal_(out[r], psi, wl.sigma * scale, seed_for(wl.index, step, r),
                     wl.outlier_frac, wl.outlier_sigma * scale)
    if wl.inject_inf_step and step == wl.inject_inf_step:
        rank, idx = inf_index(wl, step)
        if idx < psi:
            out[rank][idx] = float("inf")
    return out


def make_master(wl: Workload, device, psi_pad: int | None = None,
                psi: int | None = None) -> torch.Tensor:
    """FP32 master weights ~N(0, master_sigma) on [0, psi), zero padding."""
    psi = wl.psi if psi is None else psi
    psi_pad = wl.psi_pad if psi_pad is None else psi_pad
    out = torch.empty(psi_pad, dtype=torch.float32, device=device)
    return fill_normal_(out, psi, wl.master_sigma, seed_for(wl.index, 0, 9))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """View a CPU bf16 tensor's storage as uint16 bit patterns (no rounding)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_numpy_grad(t: torch.Tensor) -> np.ndarray:
    """A gradient buffer as the oracle takes it: uint16 bits for BF16,
    float32 for FP32 (a byte copy, no arithmetic)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()
