"""Seeded synthetic inputs and the benchmark workloads (shapes only).

This module holds none of the method's arithmetic: it draws random tensors and
names shapes. It is the one module that both the CUDA path's tests and the
oracle's tests take inputs from.

Recipe (the kernel benchmarks on the pages are synthetic fixed shapes, Table 2
and Table 7 of Mixture-of-Depths Attention):
  * tensors are drawn in the order q, k, v, kd, vd from ONE generator seeded
    with ``seed`` (0 unless stated), each element float32 N(0, 1);
  * kd and vd are multiplied by ``depth_scale`` (0.5 for the 700M-like layer;
    a power of two, so exact) before rounding;
  * everything is rounded to bf16 with round-to-nearest-even;
  * the depth stream is drawn in its append layout [L, T, Hk, d].
On the CPU the generator is ``torch.Generator('cpu')``; on a CUDA device it is
that device's Philox generator (same seed, different stream of numbers), which
is what the large workloads use so that tens of GB are not drawn on the host.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    Hq: int
    Hk: int
    d: int
    L: int
    depth_scale: float = 1.0
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """4*d*Hq*(T(T+1)/2 + T*L): causal and valid-depth work only."""
        T = self.T
        return 4.0 * self.d * self.Hq * (T * (T + 1) / 2 + T * self.L)

    def with_L(self, L: int) -> "Workload":
        return dataclasses.replace(self, L=L, name=f"{self.name}-L{L}")

    def with_T(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name=f"{self.name}-T{T}")


# The five workloads the kernel is measured and checked on.
TINY = Workload("tiny", T=128, Hq=4, Hk=2, d=64, L=4)
LAYER_700M = Workload("700m-layer23", T=4096, Hq=16, Hk=4, d=128, L=46, depth_scale=0.5)
GQA_SWEEP = [Workload(f"gqa-sweep-G{g}", T=8192, Hq=4 * g, Hk=4, d=128, L=24)
             for g in (1, 2, 4, 8)]
DEPTH_SWEEP = [Workload(f"depth-sweep-L{l}", T=16384, Hq=16, Hk=4, d=128, L=l)
               for l in (0, 8, 24, 48, 96)]
LONG = Workload("long-64k", T=65536, Hq=16, Hk=4, d=128, L=48)
LONG_L0 = LONG.with_L(0)
# The long workload at half the length: small enough for multi-counter ncu
# captures (about 3.6 GB on the device); every stream of the forward (q, o,
# the depth rows, each KV head's K/V read once) scales with T.
LONG_32K = Workload("long-32k", T=32768, Hq=16, Hk=4, d=128, L=48)

ALL = [TINY, LAYER_700M, *GQA_SWEEP, *DEPTH_SWEEP, LONG]

# The shape of the pages' kernel-efficiency table (Table 2: B=1, d=64, G=8,
# Hq=64, Hk=8, L=64, T from 4K to 64K), for context runs of forward +
# backward; not one of the five workloads above.
TABLE2 = [Workload(f"table2-T{t}", T=t, Hq=64, Hk=8, d=64, L=64)
          for t in (4096, 8192, 16384, 32768, 65536)]


def make_inputs(w: Workload, device="cpu", seed: int | None = None):
    """Returns dict q[T,Hq,d], k[T,Hk,d], v[T,Hk,d], kd[L,T,Hk,d], vd[L,T,Hk,d] (bf16)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)

    def draw(shape, mul=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if mul != 1.0:
            x.mul_(mul)
        return x.to(torch.bfloat16)

    q = draw((w.T, w.Hq, w.d))
    k = draw((w.T, w.Hk, w.d))
    v = draw((w.T, w.Hk, w.d))
    kd = draw((w.L, w.T, w.Hk, w.d), w.depth_scale)
    vd = draw((w.L, w.T, w.Hk, w.d), w.depth_scale)
    return {"q": q, "k": k, "v": v, "kd": kd, "vd": vd}


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (no arithmetic, a reinterpretation)."""
    import numpy as np
    assert x.dtype == torch.bfloat16
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def sample_rows(T: int, Hq: int, G: int, n_random: int = 64, seed: int = 1):
    """Stratified row sample for large workloads: every head at the tile edges
    and ends of the sequence, plus ``n_random`` uniform positions (seed 1)."""
    import numpy as np
    fixed = {0, 1, G - 1, G, 31, 32, 63, 64, 127, 128, 255, 256,
             T // 2, T - 2, T - 1}
    rng = np.random.default_rng(seed)
    rand = set(int(x) for x in rng.integers(0, T, size=n_random))
    ts = sorted(t for t in fixed | rand if 0 <= t < T)
    tt = np.repeat(np.array(ts, np.int64), Hq)
    hh = np.tile(np.arange(Hq, dtype=np.int64), len(ts))
    return tt, hh


@dataclasses.dataclass(frozen=True)
class ProjWorkload:
    """Shape of one FFN layer's depth-KV projection: x [T, Dm] -> slot `slot`
    of the packed [Hk, T, L, d] streams."""
    name: str
    T: int
    Dm: int
    Hk: int
    d: int
    L: int
    slot: int
    seed: int = 0

    def flops(self) -> float:
        """2 * T * Dm * (2 * Hk * d): the K and V products."""
        return 2.0 * self.T * self.Dm * 2 * self.Hk * self.d


# The long workload's layer: model width Dm = Hq * d = 16 * 128, Hk = 4, L = 48,
# writing the last slot.
PROJ_LONG = ProjWorkload("kv-proj-long-64k", T=65536, Dm=2048, Hk=4, d=128, L=48, slot=47)


def make_proj_inputs(w: ProjWorkload, device="cpu", seed: int | None = None):
    """x [T,Dm] ~ N(0,1); wk, wv [Hk*d,Dm] ~ N(0,1)/sqrt(Dm); kd, vd [Hk,T,L,d]
    prefilled ~ N(0,1) (what earlier layers wrote). All bf16, drawn in the order
    x, wk, wv, kd, vd from one generator seeded with ``seed`` (default w.seed)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)

    def draw(shape, mul=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if mul != 1.0:
            x.mul_(mul)
        return x.to(torch.bfloat16)

    n = w.Hk * w.d
    x = draw((w.T, w.Dm))
    wk = draw((n, w.Dm), 1.0 / math.sqrt(w.Dm))
    wv = draw((n, w.Dm), 1.0 / math.sqrt(w.Dm))
    kd = draw((w.Hk, w.T, w.L, w.d))
    vd = draw((w.Hk, w.T, w.L, w.d))
    return {"x": x, "wk": wk, "wv": wv, "kd": kd, "vd": vd}
