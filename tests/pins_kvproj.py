"""Pins of the oracle's depth-KV projection (an FFN layer's K or V, a linear map
of the FFN's input: reading notes Sec. 二.3, summary Sec. 2.2 "write" step).

Each pin returns (error, tolerance); run_all(orc) runs all of them.
  K1  library routine: numpy's fp64 matmul of the same bf16 values, on all
      rows and on a row subset given in scrambled order;
  K2  exact integers: small-integer x and w, so every product and sum is an
      integer far below 2^53; compared with Python's exact integer arithmetic;
  K3  selection weights: w[n, c] = 1 iff c = (3n + 1) mod Dm, so
      out[t, n] = x[t, (3n + 1) mod Dm] exactly (catches a transposed or
      shifted weight index and a dropped term).
"""
import numpy as np
import torch

from sequence_depth_attention_gb300.inputs import bf16_bits


def _bf16(a):
    return bf16_bits(torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def k1_matmul(orc):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(37, 96, generator=g).to(torch.bfloat16)
    w = (torch.randn(40, 96, generator=g) / 96 ** 0.5).to(torch.bfloat16)
    ref = x.double().numpy() @ w.double().numpy().T
    out = orc.kv_proj(bf16_bits(x), bf16_bits(w))
    rows = np.array([36, 0, 17, 5], np.int64)
    sub = orc.kv_proj(bf16_bits(x), bf16_bits(w), rows)
    err = max(np.abs(out - ref).max(), np.abs(sub - ref[rows]).max())
    return err, 1e-12 * np.abs(ref).max()


def k2_integers(orc):
    rng = np.random.default_rng(12)
    x = rng.integers(-7, 8, size=(9, 70))
    w = rng.integers(-5, 6, size=(12, 70))
    exact = [[sum(int(x[t, c]) * int(w[n, c]) for c in range(70)) for n in range(12)]
             for t in range(9)]
    out = orc.kv_proj(_bf16(x), _bf16(w))
    return float(np.abs(out - np.array(exact, np.float64)).max()), 0.0


def k3_selection(orc):
    rng = np.random.default_rng(13)
    T, Dm, N = 11, 64, 48
    x = _bf16(rng.standard_normal((T, Dm)))
    w = np.zeros((N, Dm), np.float32)
    for n in range(N):
        w[n, (3 * n + 1) % Dm] = 1.0
    out = orc.kv_proj(x, _bf16(w))
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    want = xv[:, [(3 * n + 1) % Dm for n in range(N)]]
    return float(np.abs(out - want).max()), 0.0


PINS = {"K1_matmul": k1_matmul, "K2_integers": k2_integers, "K3_selection": k3_selection}


def run_all(orc):
    return {name: fn(orc) for name, fn in PINS.items()}
