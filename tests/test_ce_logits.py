"""GPU parity of the cross-entropy on materialised logits (flce_cross_entropy)
against the fp64 oracle_ce_logits: bf16 and fp32 logits, softcap and output
multiplier, mean / sum / none reductions, ragged vocabularies, strided rows,
ignored rows. Same tolerances as the fused path (loss 2e-3 relative, gradient
max-abs 1e-2 of max|ref|, argmax exact off near-ties)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import oracle_ce_logits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _logits(N, V, seed, dtype, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((N, V), generator=g) * scale).to(dtype)


def _check(out, ref, y, what):
    valid = y.numpy() != -100
    if ref["n_valid"]:
        assert abs(float(out["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"]), (what, float(out["loss"]),
                                                                                   ref["loss"])
    rl = out["row_loss"].reshape(-1).cpu().double().numpy()
    assert np.abs(rl - ref["row_loss"]).max() <= 2e-3 * max(np.abs(ref["row_loss"]).max(), 1e-30), what
    assert np.all(rl[~valid] == 0.0)
    pred = out["predicted"].reshape(-1).cpu().numpy()
    near = ref["top2_gap"] < 1e-3
    assert np.all((pred == ref["predicted"]) | near), what
    if out["grad_logits"] is not None:
        g = out["grad_logits"].reshape(ref["grad_logits"].shape).cpu().double().numpy()
        scale = np.abs(ref["grad_logits"]).max()
        assert np.abs(g - ref["grad_logits"]).max() <= 1e-2 * max(scale, 1e-30), what


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("case", [
    dict(N=300, V=5000),
    dict(N=129, V=2049, softcap=30.0, out_mult=0.5),            # one column past a 2048 tile
    dict(N=64, V=7, softcap=2.0),                                # vocab smaller than one vector
    dict(N=500, V=4099, reduction="sum", grad_scale=0.5),
    dict(N=256, V=3000, reduction="none", row_scale=True, softcap=10.0),
])
def test_ce_logits_parity(flce, dtype, case):
    c = dict(case)
    N, V = c.pop("N"), c.pop("V")
    x = _logits(N, V, N + V, dtype)
    y = workloads.make_labels(N, V, N, 0.1)
    rs = torch.randn(N, generator=torch.Generator().manual_seed(3)) if c.pop("row_scale", False) else None
    out = flce.flce_cross_entropy(x.to(DEV), y.to(DEV), row_scale=None if rs is None else rs.to(DEV), **c)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = oracle_ce_logits(x, y, row_scale=None if rs is None else rs.double().numpy(), **c)
    _check(out, ref, y, f"{case} {dtype}")


def test_ce_logits_strided_rows_and_in_place_grad(flce):
    N, V, ld = 200, 1000, 1032
    big = _logits(N, ld, 5, torch.bfloat16)
    x = big[:, :V]                                   # row stride 1032
    y = workloads.make_labels(N, V, 5, 0.1)
    ref = oracle_ce_logits(x, y, softcap=5.0)
    out = flce.flce_cross_entropy(x.to(DEV), y.to(DEV), softcap=5.0)
    torch.cuda.synchronize()
    _check(out, ref, y, "strided")
    xd = x.to(DEV).contiguous()
    out2 = flce.flce_cross_entropy(xd, y.to(DEV), softcap=5.0, grad_in_place=True)
    torch.cuda.synchronize()
    assert out2["grad_logits"].data_ptr() == xd.data_ptr()
    _check(out2, ref, y, "in place")


def test_ce_logits_all_ignored_and_bad_label(flce):
    N, V = 64, 900
    x = _logits(N, V, 6, torch.float32)
    y = torch.full((N,), -100, dtype=torch.int64)
    out = flce.flce_cross_entropy(x.to(DEV), y.to(DEV))
    torch.cuda.synchronize()
    assert float(out["loss"]) == 0.0 and torch.all(out["grad_logits"] == 0)
    y[3] = V
    flce.flce_cross_entropy(x.to(DEV), y.to(DEV))
    assert flce.flce_get_status() & 16


def test_ce_logits_llama_vocab_rows(flce):
    """A Llama-sized vocabulary (128256) in bf16, 1024 rows, several chunks."""
    N, V = 1024, 128256
    x = _logits(N, V, 7, torch.bfloat16, scale=1.28)
    y = workloads.make_labels(N, V, 7, 0.05)
    out = flce.flce_cross_entropy(x.to(DEV), y.to(DEV), chunk_rows=384)
    torch.cuda.synchronize()
    ref = oracle_ce_logits(x, y)
    _check(out, ref, y, "llama vocab")


def _fuzz_cases(n=24, seed=77):
    rng = np.random.default_rng(seed)
    return [dict(N=int(rng.integers(1, 500)), V=int(rng.integers(2, 20000)),
                 softcap=float(rng.choice([0.0, 2.0, 30.0])), out_mult=float(rng.choice([1.0, 0.5, -1.0])),
                 reduction=str(rng.choice(["mean", "sum", "none"])), bf16=bool(rng.integers(0, 2)),
                 ign=float(rng.choice([0.0, 0.2])), seed=i) for i in range(n)]


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"N{c['N']}-V{c['V']}-{c['reduction']}")
def test_ce_logits_fuzzed(flce, case):
    """Seeded random shapes (V anywhere, including inside the 8-column vectors
    and across 8192-column tiles), dtypes, softcaps, multipliers, reductions and
    ignore fractions, against the oracle."""
    c = dict(case)
    N, V, ign, seed = c.pop("N"), c.pop("V"), c.pop("ign"), c.pop("seed")
    dtype = torch.bfloat16 if c.pop("bf16") else torch.float32
    x = _logits(N, V, 900 + seed, dtype)
    y = workloads.make_labels(N, V, 900 + seed, ign)
    out = flce.flce_cross_entropy(x.to(DEV), y.to(DEV), **c)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = oracle_ce_logits(x, y, **c)
    _check(out, ref, y, f"fuzz {case}")
