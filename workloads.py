"""Seeded synthetic inputs for the fused linear cross-entropy (FLCE) workloads.

This module only draws random numbers. It holds none of the loss arithmetic, so
both the CPU oracle (through the tests) and the CUDA path can be fed the very
same bf16 bits from it.

The five head shapes follow the LM heads the Liger-Kernel commit pages
benchmark ("Muse Glimmer" support, section Memory: hidden 6656, vocab 202048;
DeepSeek-V3 support, section Memory: hidden 7168, vocab 129280), a Llama-style
head (hidden 4096, vocab 128256), and the SpecForge DSpine page's flattened
frozen draft-proposal projection (section Changes: proposal rows flattened,
the frozen vocabulary projection applied, the shape restored).

Recipe (fixed so results are reproducible bit for bit):
  * h ~ N(0, 1) drawn in fp32, rounded to bf16 (round to nearest even);
  * W ~ N(0, 0.02^2) drawn in fp32, rounded to bf16;
  * labels uniform in [0, V), or Zipf(s) with p(k) ~ (k+1)^-s sampled by
    inverse CDF (token id = rank);
  * exactly round(frac * N) rows set to the ignore index, picked by a seeded
    permutation;
  * one torch CPU generator per tensor, seeded seed*16 + {1: h, 2: W, 3: labels,
    4: ignore mask}.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import numpy as np
import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_rows: int
    hidden: int
    vocab: int
    ignore_frac: float
    softcap: float = 0.0
    out_mult: float = 1.0
    labels: str = "uniform"        # "uniform" | "zipf"
    zipf_s: float = 1.1
    mode: str = "fwd_bwd"          # "fwd_bwd" | "ce_only" | "fwd_grad_h"
    return_predicted: bool = False
    row_shape: Optional[Tuple[int, ...]] = None   # per-row output shape, e.g. (B, k, S)
    seed: int = 0

    @property
    def flops(self) -> float:
        """Algorithmic tensor-core work of one pass: 2NHV per GEMM on the path."""
        per_gemm = 2.0 * self.n_rows * self.hidden * self.vocab
        return {"fwd_bwd": 3, "ce_only": 1, "fwd_grad_h": 2}[self.mode] * per_gemm


WORKLOADS = {
    "tiny": Workload("tiny", 256, 512, 4096, 0.10, seed=0),
    "llama": Workload("llama", 8192, 4096, 128256, 0.05, seed=1),
    "muse": Workload("muse", 8192, 6656, 202048, 0.05, softcap=30.0, out_mult=0.5,
                     return_predicted=True, seed=2),
    "dsv3": Workload("dsv3", 32768, 7168, 129280, 0.03, labels="zipf", zipf_s=1.1, seed=3),
    "frozen_ce": Workload("frozen_ce", 131072, 4096, 151936, 0.10, mode="ce_only",
                          row_shape=(16, 4, 2048), seed=4),
    "frozen_grad_h": Workload("frozen_grad_h", 131072, 4096, 151936, 0.10, mode="fwd_grad_h",
                              row_shape=(16, 4, 2048), seed=4),
}


def _gen(seed: int, slot: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 16 + slot)
    return g


def make_hidden(n_rows: int, hidden: int, seed: int) -> torch.Tensor:
    """h [N, H] bf16, N(0,1) rounded to bf16. Drawn in row blocks to bound host memory."""
    g = _gen(seed, 1)
    out = torch.empty((n_rows, hidden), dtype=torch.bfloat16)
    step = max(1, (1 << 26) // max(hidden, 1))
    for r0 in range(0, n_rows, step):
        r1 = min(n_rows, r0 + step)
        out[r0:r1] = torch.randn((r1 - r0, hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_weight(vocab: int, hidden: int, seed: int, std: float = 0.02) -> torch.Tensor:
    """W [V, H] bf16, N(0, std^2) rounded to bf16. Drawn in row blocks."""
    g = _gen(seed, 2)
    out = torch.empty((vocab, hidden), dtype=torch.bfloat16)
    step = max(1, (1 << 26) // max(hidden, 1))
    for r0 in range(0, vocab, step):
        r1 = min(vocab, r0 + step)
        out[r0:r1] = (torch.randn((r1 - r0, hidden), generator=g, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def make_labels(n_rows: int, vocab: int, seed: int, ignore_frac: float,
                kind: str = "uniform", zipf_s: float = 1.1,
                ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """labels [N] int64: uniform or Zipf ids, with exactly round(frac*N) ignored rows."""
    g = _gen(seed, 3)
    if kind == "uniform":
        lab = torch.randint(0, vocab, (n_rows,), generator=g, dtype=torch.int64)
    elif kind == "zipf":
        ranks = np.arange(1, vocab + 1, dtype=np.float64)
        p = ranks ** (-zipf_s)
        cdf = np.cumsum(p)
        cdf /= cdf[-1]
        u = torch.rand((n_rows,), generator=g, dtype=torch.float64).numpy()
        idx = np.searchsorted(cdf, u, side="right")
        lab = torch.from_numpy(np.minimum(idx, vocab - 1).astype(np.int64))
    else:
        raise ValueError(f"unknown label distribution {kind!r}")
    n_ign = int(round(ignore_frac * n_rows))
    if n_ign > 0:
        perm = torch.randperm(n_rows, generator=_gen(seed, 4))[:n_ign]
        lab[perm] = ignore_index
    return lab


def make_inputs(w: Workload, n_rows: Optional[int] = None):
    """(h, W, labels) on the CPU for a workload; n_rows overrides N (same H, V, recipe)."""
    n = w.n_rows if n_rows is None else n_rows
    h = make_hidden(n, w.hidden, w.seed)
    W = make_weight(w.vocab, w.hidden, w.seed)
    labels = make_labels(n, w.vocab, w.seed, w.ignore_frac, w.labels, w.zipf_s)
    return h, W, labels


def sample_indices(n: int, k: int, seed: int, must_include=()) -> np.ndarray:
    """A seeded sorted sample of k distinct indices in [0, n), plus must_include."""
    rng = np.random.default_rng(seed)
    k = min(k, n)
    base = rng.choice(n, size=k, replace=False)
    extra = np.asarray([i for i in must_include if 0 <= i < n], dtype=np.int64)
    return np.unique(np.concatenate([base.astype(np.int64), extra]))


def zipf_head_ids(vocab: int, k: int) -> list:
    """The k most frequent ids under the Zipf recipe (ids 0..k-1)."""
    return list(range(min(k, vocab)))


def plant_labels(labels: torch.Tensor, predicted, frac: float, seed: int,
                 ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """Labels with a seeded `frac` of the non-ignored rows replaced by the given
    predicted ids (ignored rows stay ignored). With the oracle's predictions this
    makes a batch whose token accuracy is far from the ~1/V of uniform labels."""
    lab = labels.clone()
    valid = np.nonzero(lab.numpy() != ignore_index)[0]
    k = int(round(frac * len(valid)))
    rng = np.random.default_rng(seed)
    pick = np.sort(rng.choice(valid, size=k, replace=False)) if k > 0 else np.zeros(0, np.int64)
    pred = np.asarray(predicted, dtype=np.int64)
    lab[torch.from_numpy(pick)] = torch.from_numpy(pred[pick])
    return lab


def tensor_sha256(t: torch.Tensor) -> str:
    """sha256 of a CPU tensor's raw bytes (bf16 as its 16-bit patterns)."""
    import hashlib
    x = t.contiguous()
    if x.dtype == torch.bfloat16:
        x = x.view(torch.int16)
    return hashlib.sha256(x.numpy().tobytes()).hexdigest()
