"""Seeded synthetic inputs for the lm_head logits workloads.

This module only draws random numbers; it holds none of the method's
arithmetic.  It is shared by the tests, the bench and the smoke check, which
hand the same tensors to the CUDA path and to the CPU oracle.

Workload shapes follow the pages:
  * 50304 x 512 W4-g64 and 151936 x 1024 W4-g64 / W8-g128 -- "Fused WNA16
    GEMM for tied quantized lm_head logits", Perf evals table;
  * 151936 x 2048 int8 per-row + fp16 reference, top-8 rescoring -- same
    page, reviewer comment items 1-2 (Qwen2.5-Coder-3B tied head);
  * 248320 x 5120 int4 g128 bf16 scales, MSE clip -- radiance_lmhead_int4.py
    module docstring.
Weights are N(0, 0.02) drawn in fp32 and cast to the storage dtype;
activations are N(0, 1) cast to the activation dtype.  The captured decode
states the pages measured on are not available; these rows stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

F32, F16, BF16 = 0, 1, 2
TORCH_DTYPE = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
RTN, MSE = 0, 1


@dataclass(frozen=True)
class Workload:
    name: str
    n: int                 # vocab rows
    k: int                 # hidden size
    bits: int              # 4 or 8
    group: int             # 64, 128 or 0 (= one scale per row)
    scale_dtype: int       # F16 or BF16
    clip: int              # RTN or MSE
    w_dtype: int           # dtype the unquantised weight is held in
    x_dtype: int           # activation / logits dtype
    ms: tuple = (1,)       # token counts the workload is run at
    w_seed: int = 0
    x_seed: int = 1
    x_continues_w: bool = False   # draw X from the generator after W
    rows: int = 0          # number of independent M=1 rows (argmax study)
    rescore_k: int = 0     # top-K rescoring width (0 = none)
    notes: tuple = field(default_factory=tuple)


WORKLOADS = {
    "pr_fixture_50304x512_w4g64": Workload(
        "pr_fixture_50304x512_w4g64", 50304, 512, 4, 64, F16, RTN, F32, F16,
        ms=(1,), w_seed=0, x_continues_w=True),
    "qwen_151936x1024_w4g64": Workload(
        "qwen_151936x1024_w4g64", 151936, 1024, 4, 64, F16, RTN, F32, F16,
        ms=(1, 32, 256)),
    "qwen_151936x1024_w8g128": Workload(
        "qwen_151936x1024_w8g128", 151936, 1024, 8, 128, F16, RTN, F32, F16,
        ms=(1, 32, 256)),
    "qwen_151936x2048_w8row_rescore": Workload(
        "qwen_151936x2048_w8row_rescore", 151936, 2048, 8, 0, F16, RTN, F16, F16,
        ms=(1,), x_seed=2, rows=4096, rescore_k=8),
    "head_248320x5120_w4g128_mse": Workload(
        "head_248320x5120_w4g128_mse", 248320, 5120, 4, 128, BF16, MSE, BF16, BF16,
        ms=(1, 2, 3, 4, 5, 16)),
}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weight(n: int, k: int, dtype: int, seed: int = 0, device="cpu",
           gen: torch.Generator | None = None) -> torch.Tensor:
    """W ~ N(0, 0.02) drawn in fp32, then cast to `dtype`."""
    g = gen if gen is not None else generator(seed, device)
    w = torch.randn(n, k, generator=g, dtype=torch.float32, device=device)
    w.mul_(0.02)
    return w.to(TORCH_DTYPE[dtype])


def activations(m: int, k: int, dtype: int, seed: int = 1, device="cpu",
                gen: torch.Generator | None = None) -> torch.Tensor:
    """X ~ N(0, 1) drawn in fp32, then cast to `dtype`."""
    g = gen if gen is not None else generator(seed, device)
    x = torch.randn(m, k, generator=g, dtype=torch.float32, device=device)
    return x.to(TORCH_DTYPE[dtype])


def bias(n: int, dtype: int, seed: int = 3, device="cpu") -> torch.Tensor:
    g = generator(seed, device)
    b = torch.randn(n, generator=g, dtype=torch.float32, device=device)
    return b.mul_(0.1).to(TORCH_DTYPE[dtype])


def workload_tensors(wl: Workload, m: int, device="cpu"):
    """(W, X) for workload `wl` at M = m, seeded as the workload states."""
    if wl.x_continues_w:
        g = generator(wl.w_seed, device)
        w = weight(wl.n, wl.k, wl.w_dtype, device=device, gen=g)
        x = activations(m, wl.k, wl.x_dtype, device=device, gen=g)
        return w, x
    w = weight(wl.n, wl.k, wl.w_dtype, seed=wl.w_seed, device=device)
    x = activations(m, wl.k, wl.x_dtype, seed=wl.x_seed, device=device)
    return w, x


def random_nibbles(n: int, k: int, seed: int = 5) -> torch.Tensor:
    g = generator(seed, "cpu")
    return torch.randint(0, 16, (n, k), generator=g, dtype=torch.uint8)
