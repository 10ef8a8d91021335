"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers and shapes them; it holds none of the
layer's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any of the method.

Recipe (the same for every workload):
  * q, k, v ~ N(0, 1); q and k are L2-normalised per (token, head) over the
    key dimension in fp32, then every tensor is rounded to bf16;
  * beta = sigmoid(N(0, 1)) rounded to bf16;
  * log_alpha = -5 * sigmoid(N(mu, 1)) per key channel, rounded to bf16, so it
    lies in [-5, 0] (mu = 0, or 2 for decay concentrated near the bound);
  * initial state ~ N(0, std^2) in fp32 (std = 0.02) or zeros;
  * draws happen in the order q, k, v, beta-logits, decay-logits, state.

Small problems are drawn on the host with numpy's PCG64 generator (portable
and reproducible); large ones are drawn on the device with torch's generator
so that a 1M-token problem does not go through host memory.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One named problem shape (sizes only; no arithmetic)."""

    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    seed: int
    decay_mean: float = 0.0
    init_std: float = 0.0
    out_dtype: torch.dtype = torch.bfloat16
    seqlens: tuple = field(default=())  # packed sequences when non-empty

    @property
    def tokens(self) -> int:
        return self.B * self.T


def varlen_lengths(total: int, n: int, seed: int) -> list[int]:
    """n lengths summing to `total`: n-1 distinct cut points drawn uniformly
    from {1, ..., total-1}, sorted, and differenced."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, total), size=n - 1, replace=False))
    edges = np.concatenate([[0], cuts, [total]])
    return [int(x) for x in np.diff(edges)]


WORKLOADS = {
    # fp32 output and final state, zero initial state, d = 64
    "tiny": Workload("tiny", 1, 256, 2, 64, 64, seed=0, out_dtype=torch.float32),
    "prefill_8k": Workload("prefill_8k", 1, 8192, 32, 128, 128, seed=1, init_std=0.02),
    "varlen_64k": Workload("varlen_64k", 1, 65536, 32, 128, 128, seed=2,
                           seqlens=tuple(varlen_lengths(65536, 4, 2))),
    "long_1m": Workload("long_1m", 1, 1 << 20, 16, 128, 128, seed=3, decay_mean=2.0),
    "decode": Workload("decode", 256, 1, 32, 128, 128, seed=4, init_std=0.02),
    "prefill_64k": Workload("prefill_64k", 1, 65536, 32, 128, 128, seed=1, init_std=0.02),
}


def _sigmoid_np(x):
    return 1.0 / (1.0 + np.exp(-x))


def _l2n_np(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True))


def make_inputs(B, T, H, dk, dv, seed, decay_mean=0.0, init_std=0.0, n_states=None,
                device="cpu"):
    """Return dict(q, k, v, log_alpha, beta, initial_state) as torch tensors.

    Shapes: q, k, log_alpha [B,T,H,dk] bf16; v [B,T,H,dv] bf16; beta [B,T,H]
    bf16; initial_state [n_states or B, H, dk, dv] fp32 or None when
    init_std == 0.  device="cpu" draws with numpy; a CUDA device draws with
    torch's generator on that device.
    """
    n_states = B if n_states is None else n_states
    if str(device) == "cpu":
        rng = np.random.default_rng(seed)
        f32 = np.float32
        q = _l2n_np(rng.standard_normal((B, T, H, dk), dtype=f32))
        k = _l2n_np(rng.standard_normal((B, T, H, dk), dtype=f32))
        v = rng.standard_normal((B, T, H, dv), dtype=f32)
        beta = _sigmoid_np(rng.standard_normal((B, T, H), dtype=f32))
        la = -5.0 * _sigmoid_np(rng.standard_normal((B, T, H, dk), dtype=f32) + f32(decay_mean))
        s0 = (rng.standard_normal((n_states, H, dk, dv), dtype=f32) * f32(init_std)
              if init_std > 0 else None)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
        out = dict(q=t(q), k=t(k), v=t(v), log_alpha=t(la), beta=t(beta),
                   initial_state=None if s0 is None else torch.from_numpy(s0.astype(np.float32)))
        return out
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    def l2n_bf16(shape):
        # in place, in slabs along T, to bound the fp32 temporaries
        x = normal(shape)
        x /= x.norm(dim=-1, keepdim=True)
        return x.to(torch.bfloat16)

    q = l2n_bf16((B, T, H, dk))
    k = l2n_bf16((B, T, H, dk))
    v = normal((B, T, H, dv)).to(torch.bfloat16)
    beta = torch.sigmoid(normal((B, T, H))).to(torch.bfloat16)
    x = normal((B, T, H, dk))
    x += decay_mean
    la = (torch.sigmoid_(x) * -5.0).to(torch.bfloat16)
    del x
    s0 = normal((n_states, H, dk, dv)) * init_std if init_std > 0 else None
    return dict(q=q, k=k, v=v, log_alpha=la, beta=beta, initial_state=s0)


def workload_inputs(w: Workload, device="cpu", T=None):
    """Inputs for a named workload (optionally truncated to T tokens)."""
    T = w.T if T is None else T
    n_states = len(w.seqlens) if w.seqlens else w.B
    return make_inputs(w.B, T, w.H, w.dk, w.dv, w.seed, w.decay_mean, w.init_std,
                       n_states=n_states, device=device)


def cu_seqlens_of(lengths) -> torch.Tensor:
    """Offsets [0, l0, l0+l1, ...] as int32 (a prefix sum of sizes, no method arithmetic)."""
    return torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
