"""Seeded synthetic inputs for the five workloads (no attention arithmetic).

Recipe, per workload: a torch.Generator on the target device seeded with
``seed``; tensors are drawn in the order q, k, v, d_o, then any extra draws
(the heavy-row selection); each draw is float32, scaled as the workload says,
then rounded once to the kernel dtype.  Large key/value caches are drawn one
batch row at a time to bound the float32 scratch.  The same call on the same
device type returns the same values, so the oracle (on the host) and the
CUDA path see identical inputs.

Workloads (the sizes of the long-sequence settings the methods are measured on):
  tiny_fp32_causal         fp32 causal, B=1 H=2 N=256 d=64, chunks of 64
  causal_32k_ring          bf16 causal, B=1 H=32 N=32768 d=128, chunks of 4096
  causal_128k_balanced     bf16 causal, B=1 H=32 N=131072 d=128, chunks of 4096
  decode_gqa_1m            bf16, B=8 Hq=32 Hkv=8, 1 query, N=1048576 keys, d=128
  noncausal_64k_heavytail  bf16 non-causal, B=2 H=16 N=65536 d=64, 1% of the
                           key rows of every (b, h) scaled by 8
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    chunk: int
    causal: bool
    dtype: torch.dtype
    seed: int
    qk_amp: float = 1.0      # q and k ~ qk_amp * N(0, 1)
    v_amp: float = 1.0       # v ~ v_amp * N(0, 1) (or U(-1, 1))
    v_uniform: bool = False
    heavy_frac: float = 0.0  # fraction of key rows per (b, h) multiplied ...
    heavy_mult: float = 1.0  # ... by this factor before rounding
    decode: bool = False     # one query token per sequence

    @property
    def Nq(self) -> int:
        return 1 if self.decode else self.N

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in (
        Workload("tiny_fp32_causal", 1, 2, 2, 256, 64, 64, True, torch.float32, 1001),
        Workload("causal_32k_ring", 1, 32, 32, 32768, 128, 4096, True, torch.bfloat16, 1002,
                 qk_amp=0.5, v_amp=0.5),
        Workload("causal_128k_balanced", 1, 32, 32, 131072, 128, 4096, True, torch.bfloat16,
                 1003, qk_amp=0.5, v_amp=0.5),
        Workload("decode_gqa_1m", 8, 32, 8, 1048576, 128, 4096, False, torch.bfloat16, 1004,
                 decode=True),
        Workload("noncausal_64k_heavytail", 2, 16, 16, 65536, 64, 4096, False, torch.bfloat16,
                 1005, qk_amp=2.0, v_uniform=True, heavy_frac=0.01, heavy_mult=8.0),
    )
}


def _randn(shape, gen, device, amp, dtype, rows_at_once=False):
    if not rows_at_once:
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * amp).to(dtype)
    out = torch.empty(shape, dtype=dtype, device=device)
    for b in range(shape[0]):
        out[b] = (torch.randn(shape[1:], generator=gen, device=device,
                              dtype=torch.float32) * amp).to(dtype)
    return out


def make_inputs(w: Workload | str, device="cpu", with_grad=True, seed=None):
    """Returns dict(q, k, v, d_o[, heavy_rows]) for workload ``w``."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    big = w.B * w.Hkv * w.N * w.D > (1 << 31)
    q = _randn((w.B, w.Hq, w.Nq, w.D), gen, device, w.qk_amp, torch.float32)
    k = _randn((w.B, w.Hkv, w.N, w.D), gen, device, w.qk_amp, torch.float32 if w.heavy_frac else w.dtype,
               rows_at_once=big)
    if w.v_uniform:
        v = (torch.rand((w.B, w.Hkv, w.N, w.D), generator=gen, device=device) * 2.0 - 1.0).to(w.dtype)
    else:
        v = _randn((w.B, w.Hkv, w.N, w.D), gen, device, w.v_amp, w.dtype, rows_at_once=big)
    out = {"q": q.to(w.dtype), "v": v}
    if with_grad:
        out["d_o"] = _randn((w.B, w.Hq, w.Nq, w.D), gen, device, 1.0, w.dtype)
    if w.heavy_frac:
        n_heavy = int(w.heavy_frac * w.N)
        rows = torch.empty((w.B, w.Hkv, n_heavy), dtype=torch.int64, device=device)
        for b in range(w.B):
            for h in range(w.Hkv):
                sel = torch.randperm(w.N, generator=gen, device=device)[:n_heavy]
                rows[b, h] = sel
                k[b, h, sel] *= w.heavy_mult
        out["heavy_rows"] = rows
        k = k.to(w.dtype)
    out["k"] = k
    return out


def to_f64_numpy(t: torch.Tensor):
    """Exact upcast of the values a kernel sees, for the host oracle."""
    return t.detach().to("cpu", torch.float64).numpy()


def random_tensor(shape, seed, amp=1.0, dtype=torch.bfloat16, device="cpu",
                  uniform=False):
    """One seeded draw (float32 N(0,1) * amp or U(-amp, amp)) rounded to dtype."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if uniform:
        x = (torch.rand(shape, generator=gen, device=device) * 2.0 - 1.0) * amp
    else:
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * amp
    return x.to(dtype)
