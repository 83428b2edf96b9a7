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

Recipe (fixed so that results are reproducible bit for bit, on any machine):
  * every random number comes from a counter-based generator: SplitMix64
    (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014) applied to key + (i + 1) * 0x9E3779B97F4A7C15 for the i-th
    draw of a tensor. Only 64-bit integer arithmetic, so the same bits come out
    on x86 and Arm (torch's own normal sampler does not: its vectorised paths
    differ between the two);
  * h ~ N(0, 1): Box-Muller in fp64 on pairs of 53-bit uniforms (element 2k
    takes the cosine, 2k + 1 the sine), rounded to fp32, then to bf16 (round to
    nearest even);
  * W ~ N(0, 0.02^2): the same normals times 0.02 in fp64, then fp32, then bf16;
  * labels uniform in [0, V) (the top 32 bits of a draw times V, shifted down
    32), or Zipf(s) with p(k) ~ (k+1)^-s sampled by inverse CDF (token id =
    rank);
  * exactly round(frac * N) rows set to the ignore index: the rows with the
    smallest draws of their own stream;
  * one stream per tensor, keyed seed*16 + {1: h, 2: W, 3: labels, 4: ignore
    mask}.
The fp64 log, sqrt, cos and sin of Box-Muller may differ by an ulp between
math libraries; a bf16 result changes only when the fp64 value lies within
that ulp of a bf16 rounding midpoint (about 1e-13 per element). The tests that
compare with stored oracle results check a hash of the inputs first.
"""
from __future__ import annotations

import dataclasses
import functools
import os
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
    # the DeepSeek-V3 training head returns the predicted tokens beside the token
    # accuracy (Liger-Kernel DeepSeek-V3 support, Summary: lce_forward's output)
    "dsv3": Workload("dsv3", 32768, 7168, 129280, 0.03, labels="zipf", zipf_s=1.1, return_predicted=True, seed=3),
    "frozen_ce": Workload("frozen_ce", 131072, 4096, 151936, 0.10, mode="ce_only",
                          row_shape=(16, 4, 2048), seed=4),
    "frozen_grad_h": Workload("frozen_grad_h", 131072, 4096, 151936, 0.10, mode="fwd_grad_h",
                              row_shape=(16, 4, 2048), seed=4),
}


_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22            # elements per generation task


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64's output function on uint64 (wrapping arithmetic)."""
    z = z ^ (z >> np.uint64(30))
    z = z * _MIX1
    z = z ^ (z >> np.uint64(27))
    z = z * _MIX2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, slot: int) -> np.uint64:
    return _mix(np.asarray([seed * 16 + slot], dtype=np.uint64) * _GAMMA)[0]


def draws(key: np.uint64, i0: int, n: int) -> np.ndarray:
    """Draws i0 .. i0+n-1 of the stream `key`: uint64 [n]."""
    i = np.arange(i0 + 1, i0 + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * _GAMMA)


def _normals_block(key: np.uint64, i0: int, n: int, scale: float) -> np.ndarray:
    """Normals i0 .. i0+n-1 of the stream (Box-Muller on draw pairs), times
    scale, as fp32."""
    k0, k1 = i0 // 2, (i0 + n + 1) // 2
    d = draws(key, 2 * k0, 2 * (k1 - k0))
    u1 = ((d[0::2] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53   # (0, 1]
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53                    # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    t = (2.0 * np.pi) * u2
    z = np.empty(2 * (k1 - k0))
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    z = z[i0 - 2 * k0:i0 - 2 * k0 + n]
    if scale != 1.0:
        z = z * scale
    return z.astype(np.float32)


def _normal_bf16(shape, key: np.uint64, scale: float) -> torch.Tensor:
    """A bf16 tensor of normals (row-major element index = draw index),
    generated in blocks on a thread pool (numpy releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def job(i0):
        m = min(_BLOCK, n - i0)
        out[i0:i0 + m] = _normals_block(key, i0, m, scale)

    with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        list(ex.map(job, range(0, n, _BLOCK)))
    return torch.from_numpy(out).view(*shape).to(torch.bfloat16)


@functools.lru_cache(maxsize=4)
def _cached_normal_bf16(shape, seed: int, slot: int, scale: float) -> torch.Tensor:
    return _normal_bf16(shape, _key(seed, slot), scale)


def make_hidden(n_rows: int, hidden: int, seed: int) -> torch.Tensor:
    """h [N, H] bf16, N(0,1) rounded to bf16. Row i of a smaller N equals row i
    of a larger one. (A fresh copy of a small per-process cache: a full-size
    head takes seconds to draw.)"""
    return _cached_normal_bf16((n_rows, hidden), seed, 1, 1.0).clone()


def make_weight(vocab: int, hidden: int, seed: int, std: float = 0.02) -> torch.Tensor:
    """W [V, H] bf16, N(0, std^2) rounded to bf16 (a fresh copy, as make_hidden)."""
    return _cached_normal_bf16((vocab, hidden), seed, 2, float(std)).clone()


def make_labels(n_rows: int, vocab: int, seed: int, ignore_frac: float,
                kind: str = "uniform", zipf_s: float = 1.1,
                ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """labels [N] int64: uniform or Zipf ids, with exactly round(frac*N) ignored rows."""
    d = draws(_key(seed, 3), 0, n_rows)
    if kind == "uniform":
        lab = (((d >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)).astype(np.int64)
    elif kind == "zipf":
        ranks = np.arange(1, vocab + 1, dtype=np.float64)
        p = ranks ** (-zipf_s)
        cdf = np.cumsum(p)
        cdf /= cdf[-1]
        u = (d >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        idx = np.searchsorted(cdf, u, side="right")
        lab = np.minimum(idx, vocab - 1).astype(np.int64)
    else:
        raise ValueError(f"unknown label distribution {kind!r}")
    n_ign = int(round(ignore_frac * n_rows))
    if n_ign > 0:
        order = np.argsort(draws(_key(seed, 4), 0, n_rows), kind="stable")
        lab[order[:n_ign]] = ignore_index
    return torch.from_numpy(lab)


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
