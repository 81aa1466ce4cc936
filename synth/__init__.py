"""Seeded synthetic inputs for the serial Markov draft walk.

This module only draws random tensors of the right shapes and distributions;
it holds none of the walk's arithmetic.  Both the CUDA path's tests and the
CPU oracle consume what it returns, so the two sides always see identical
inputs.

The pages measure the walk inside SGLang and vLLM serving runs on released
checkpoints and datasets; none of those are available here, so seeded tensors
of the same shapes stand in for them:

* W1 [V, r] ~ N(0, 1) / 16 and W2 [V, r] ~ N(0, 1), so W2 @ W1[p] ~ N(0, 1);
* base logits [B, gamma, V] ~ N(0, sigma^2);
* anchors uniform in [0, V); temperatures per request;
* a recurrent head's matrix M [r, r] ~ N(0, 1) / 16 (``make_cell_matrix``; [3r, r]
  for the GRU), so M @ h is of the size of the W1 rows it is added to, and the
  GRU's token tables [3, V, r] ~ N(0, 1) / 16 (``make_cell_tables``).

Every tensor is drawn in fp32 from ``torch.Generator('cpu')`` and rounded to
bf16 by PyTorch's cast: W1 then W2 from the config's weight seed, then base
and anchor from a per-round seed.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

RANK = 256


@dataclass(frozen=True)
class WalkConfig:
    """One workload: vocabulary, rank, walk length, batch sizes, sampling."""
    name: str
    V: int
    gamma: int
    batches: List[int]
    seed: int
    base_std: float = 1.0
    spike: float = 0.0            # added to one uniform token per (request, step)
    temperatures: tuple = (0.0,)  # request b uses temperatures[b % len]
    noise_seed: int = 0
    r: int = RANK
    rounds: int = 1               # distinct (base, anchor) rounds per weight set
    note: str = ""


CONFIGS = {
    "tiny": WalkConfig("tiny", V=4096, gamma=4, batches=[1], seed=0,
                       note="tiny walk: V=4096, gamma=4, B=1, greedy"),
    "qwen3_resident": WalkConfig(
        "qwen3_resident", V=151936, gamma=7, batches=[1], seed=1, spike=6.0, rounds=100,
        note="Qwen3-scale fully resident walk: V=151,936, gamma=7, B=1, greedy, "
             "+6 spike at one token per step, 100 rounds"),
    "long_block": WalkConfig(
        "long_block", V=151936, gamma=16, batches=[1, 4, 8, 16], seed=2,
        note="long-block batched walk: V=151,936, gamma=16, B in {1,4,8,16}, greedy"),
    "partial": WalkConfig(
        "partial", V=248320, gamma=16, batches=[1, 8], seed=3,
        note="partial residency: V=248,320 (W2 127 MB), gamma=16, B in {1,8}, greedy"),
    "sampled": WalkConfig(
        "sampled", V=129280, gamma=5, batches=[1, 16, 64, 128, 253], seed=4,
        base_std=2.0, temperatures=(0.0, 0.6, 1.0), noise_seed=1234,
        note="sampled large-batch walk: V=129,280, gamma=5, B in {1,16,64,128,253}, "
             "T cycling {0, 0.6, 1.0}, Philox seed 1234"),
}


@dataclass
class WalkInputs:
    """One round's tensors (CPU).  bf16 tensors can be viewed as uint16 bits."""
    W1: torch.Tensor          # bf16 [V, r]
    W2: torch.Tensor          # bf16 [V, r]
    base: torch.Tensor        # bf16 [B, gamma, V]
    anchor: torch.Tensor      # int32 [B]
    temperature: torch.Tensor  # float32 [B]
    seed: int                 # Philox seed of the round
    meta: dict = field(default_factory=dict)

    @property
    def V(self):
        return self.W2.shape[0]

    @property
    def B(self):
        return self.base.shape[0]

    @property
    def gamma(self):
        return self.base.shape[1]


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a bf16 tensor as a numpy uint16 array (no copy if possible)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def make_weights(V: int, r: int, seed: int):
    """W1 ~ N(0,1)/16 and W2 ~ N(0,1), both bf16 [V, r]."""
    g = torch.Generator("cpu").manual_seed(seed)
    W1 = (torch.randn(V, r, generator=g) / 16.0).to(torch.bfloat16)
    W2 = torch.randn(V, r, generator=g).to(torch.bfloat16)
    return W1, W2, g


def make_round(g: torch.Generator, V: int, B: int, gamma: int, base_std: float,
               spike: float, temperatures, noise_seed: int):
    """base [B, gamma, V], anchor [B] and temperature [B] from generator g."""
    base = torch.randn(B, gamma, V, generator=g) * base_std
    if spike:
        pos = torch.randint(0, V, (B, gamma), generator=g)
        base.view(B * gamma, V)[torch.arange(B * gamma), pos.view(-1)] += spike
    base = base.to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    temps = torch.tensor([temperatures[b % len(temperatures)] for b in range(B)],
                         dtype=torch.float32)
    return base, anchor, temps


def round_seed(cfg, B: int, round_index: int) -> int:
    """Seed of the generator that draws one round's base, anchor and temperature."""
    return 1000 * (cfg.seed + 1) + 7919 * B + round_index


def make_inputs(cfg, B: Optional[int] = None, round_index: int = 0,
                weights=None) -> WalkInputs:
    """Inputs of one round of config ``cfg`` (a name or a WalkConfig).

    Weights come from ``cfg.seed``; the round's base, anchor and temperature
    from ``round_seed(cfg, B, round_index)``.  Pass ``weights=(W1, W2)`` to
    reuse weights already drawn for this config.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    B = cfg.batches[0] if B is None else B
    if weights is None:
        W1, W2, _ = make_weights(cfg.V, cfg.r, cfg.seed)
    else:
        W1, W2 = weights
    g = torch.Generator("cpu").manual_seed(round_seed(cfg, B, round_index))
    base, anchor, temps = make_round(g, cfg.V, B, cfg.gamma, cfg.base_std, cfg.spike,
                                     cfg.temperatures, cfg.noise_seed)
    return WalkInputs(W1, W2, base, anchor, temps, cfg.noise_seed,
                      meta={"config": cfg.name, "B": B, "round": round_index})


def make_custom(V: int, gamma: int, B: int, seed: int, r: int = RANK,
                base_std: float = 1.0, temperatures=(0.0,), noise_seed: int = 0,
                spike: float = 0.0) -> WalkInputs:
    """Inputs of an arbitrary shape with the same distributions."""
    W1, W2, g = make_weights(V, r, seed)
    base, anchor, temps = make_round(g, V, B, gamma, base_std, spike, temperatures,
                                     noise_seed)
    return WalkInputs(W1, W2, base, anchor, temps, noise_seed,
                      meta={"config": "custom", "V": V, "B": B, "seed": seed})


def make_cell_matrix(seed: int, r: int = RANK, rows: Optional[int] = None) -> torch.Tensor:
    """A recurrent head's bf16 matrix M [rows, r] ~ N(0, 1) / 16 (synthetic
    weights); rows = r, or 3r for the GRU's three gate matrices stacked."""
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(rows or r, r, generator=g) / 16).to(torch.bfloat16)


def make_cell_tables(V: int, seed: int, r: int = RANK) -> torch.Tensor:
    """The GRU head's three bf16 token tables [3, V, r] ~ N(0, 1) / 16 (the input
    projections folded into per-token rows; synthetic weights)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(3, V, r, generator=g) / 16).to(torch.bfloat16)
