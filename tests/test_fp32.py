"""GPU parity of the fp32-operand variant (h, W and grad_h in fp32; tcgen05
kind::tf32 GEMMs) against the fp64 oracle on the exact fp32 inputs. The pages
run their parity and convergence suites in fp32 as well as bf16 (Liger-Kernel
Muse Glimmer page, Testing Done; DeepSeek-V3 page, Testing Done table). Same
tolerances as the bf16 path."""
import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle
from test_parity import check_against_oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _inputs_f32(N, H, V, seed, ign=0.1, w_std=0.05):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn((N, H), generator=g)
    W = torch.randn((V, H), generator=g) * w_std
    y = workloads.make_labels(N, V, seed, ign)
    return h, W, y


# 0: per-GEMM tile choice (128-row tiles at these sizes); 32: 256-row tiles forced
@pytest.mark.parametrize("flags", [0, 32])
@pytest.mark.parametrize("case", [
    dict(N=256, H=512, V=4096),
    dict(N=300, H=192, V=1000, chunk_rows=128),
    dict(N=129, H=64, V=4100),
    dict(N=513, H=136, V=777, chunk_rows=256, softcap=30.0, out_mult=0.5),
    dict(N=256, H=256, V=2048, softcap=2.0, out_mult=0.5, reduction="sum", grad_scale=0.75),
])
def test_fp32_parity(flce, case, flags):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h, W, y = _inputs_f32(N, H, V, seed=N + H + V)
    G0 = (np.random.default_rng(2).standard_normal((V, H)) * 1e-3).astype(np.float32).astype(np.float64)
    gW = torch.from_numpy(G0).float().to(DEV)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, return_predicted=True,
                                     flags=flags, **c)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert out["grad_h"].dtype == torch.float32
    ref = flce_oracle(h, W, y, grad_W0=G0, softcap=c.get("softcap", 0.0), out_mult=c.get("out_mult", 1.0),
                      reduction=c.get("reduction", "mean"), grad_scale=c.get("grad_scale", 1.0))
    rep = check_against_oracle(out, ref, y, grad_W0=G0, what=f"fp32 {case} flags={flags}")
    print(case, flags, rep)


def test_fp32_forward_and_ce_only(flce):
    N, H, V = 400, 256, 3333
    h, W, y = _inputs_f32(N, H, V, seed=7)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    f = flce.flce_forward(hd, Wd, yd, return_lse=True, softcap=5.0)
    loss, acc = flce.flce_ce_only(hd, Wd, yd, softcap=5.0)
    torch.cuda.synchronize()
    ref = flce_oracle(h, W, y, softcap=5.0, need_grad_h=False, need_grad_W=False)
    assert float(loss) == float(f["loss"])
    assert abs(float(loss) - ref["loss"]) <= 2e-3 * ref["loss"]
    assert np.abs(f["lse"].cpu().double().numpy() - ref["lse"]).max() <= 1e-3 * np.abs(ref["lse"]).max()
    check_against_oracle({"loss": loss, "token_accuracy": acc, "predicted": f["predicted"]}, ref, y, what="fwd")


def test_fp32_frozen_weight_and_llama_width(flce):
    """A Llama-width head (H = 4096) in fp32 with a frozen W, two chunks."""
    N, H, V = 1024, 4096, 32000
    h, W, y = _inputs_f32(N, H, V, seed=8, w_std=0.02)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=None, return_predicted=True,
                                     chunk_rows=512)
    torch.cuda.synchronize()
    ref = flce_oracle(h, W, y, need_grad_W=False)
    check_against_oracle(out, ref, y, what="fp32 llama width")


def test_fp32_rejects_unsupported_modes(flce):
    h, W, y = _inputs_f32(64, 64, 300, seed=9)
    with pytest.raises(flce.FlceError):
        flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), low_memory=True)
    with pytest.raises(ValueError):
        flce.flce_forward_backward(h.to(DEV), W.to(DEV).bfloat16(), y.to(DEV))


def _fuzz_cases(n=16, seed=32):
    rng = np.random.default_rng(seed)
    return [dict(N=int(rng.integers(1, 600)), H=int(8 * rng.integers(1, 40)), V=int(rng.integers(2, 2500)),
                 softcap=float(rng.choice([0.0, 2.0, 30.0])), out_mult=float(rng.choice([1.0, 0.5, -1.5])),
                 chunk_rows=int(rng.choice([0, 128, 256])), flags=int(rng.choice([0, 16, 32])), seed=i)
            for i in range(n)]


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"N{c['N']}-H{c['H']}-V{c['V']}-f{c['flags']}")
def test_fp32_fuzzed_shapes(flce, case):
    """Seeded random shapes and options on the tf32 path, against the oracle
    on the exact fp32 inputs."""
    c = dict(case)
    N, H, V, seed = c.pop("N"), c.pop("H"), c.pop("V"), c.pop("seed")
    h, W, y = _inputs_f32(N, H, V, seed=500 + seed)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=torch.zeros(V, H, device=DEV),
                                     return_predicted=True, **c)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, softcap=c["softcap"], out_mult=c["out_mult"])
    check_against_oracle(out, ref, y, what=f"fp32 fuzz {case}")


def _rel_errs(out, ref, G0=None):
    loss = abs(float(out["loss"]) - ref["loss"]) / abs(ref["loss"])
    gh = out["grad_h"].double().cpu().numpy()
    e_h = np.abs(gh - ref["grad_h"]).max() / np.abs(ref["grad_h"]).max()
    e_w = None
    if out.get("grad_W") is not None:
        d = ref["grad_W"] - (0.0 if G0 is None else G0)
        e_w = np.abs(out["grad_W"].double().cpu().numpy() - ref["grad_W"]).max() / np.abs(d).max()
    return loss, e_h, e_w


@pytest.mark.parametrize("case", [
    dict(N=256, H=512, V=4096),
    dict(N=513, H=136, V=777, chunk_rows=256, softcap=30.0, out_mult=0.5),
    dict(N=700, H=1024, V=5000, softcap=2.0, out_mult=-1.5, reduction="sum", grad_scale=0.75),
])
def test_fp32_three_pass_reaches_fp32_accuracy(flce, case):
    """FLCE_FLAG_F32_3PASS: each product as hi*hi + hi*lo + lo*hi in tf32. The
    loss and both gradients come within fp32 rounding of the fp64 oracle on the
    exact fp32 inputs (errors of about 1e-6), two orders of magnitude closer
    than the single-pass tf32 products, whose 10-bit mantissas limit them to
    about 1e-3."""
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h, W, y = _inputs_f32(N, H, V, seed=N + H + V + 1)
    G0 = (np.random.default_rng(3).standard_normal((V, H)) * 1e-3).astype(np.float32).astype(np.float64)
    ref = flce_oracle(h, W, y, grad_W0=G0, softcap=c.get("softcap", 0.0), out_mult=c.get("out_mult", 1.0),
                      reduction=c.get("reduction", "mean"), grad_scale=c.get("grad_scale", 1.0))
    errs = {}
    for flags in (0, flce.FLCE_FLAG_F32_3PASS):
        gW = torch.from_numpy(G0).float().to(DEV)
        out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, return_predicted=True,
                                         flags=flags, **c)
        torch.cuda.synchronize()
        assert flce.flce_get_status() == 0
        check_against_oracle(out, ref, y, grad_W0=G0, what=f"fp32 {case} flags={flags}")
        errs[flags] = _rel_errs(out, ref, G0)
    l3, h3, w3 = errs[flce.FLCE_FLAG_F32_3PASS]
    l1, h1, w1 = errs[0]
    print(case, "tf32", errs[0], "3-pass", errs[flce.FLCE_FLAG_F32_3PASS])
    assert l3 <= 1e-5 and h3 <= 1e-4 and w3 <= 1e-4, errs
    assert h3 * 20 <= h1 and w3 * 20 <= w1, errs


def test_fp32_three_pass_forward_llama_width_and_host_inputs(flce):
    """The three-pass forward at H = 4096 (the lse of every row), and the same
    call with host inputs, which splits each staged chunk."""
    N, H, V = 600, 4096, 20000
    h, W, y = _inputs_f32(N, H, V, seed=11, w_std=0.02)
    f = flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV), return_lse=True, flags=flce.FLCE_FLAG_F32_3PASS)
    torch.cuda.synchronize()
    ref = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=False)
    assert np.abs(f["lse"].cpu().double().numpy() - ref["lse"]).max() <= 1e-5 * np.abs(ref["lse"]).max()
    gW = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    a = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, chunk_rows=256,
                                   flags=flce.FLCE_FLAG_F32_3PASS)
    gW2 = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    b = flce.flce_forward_backward_from_host(h.pin_memory(), W.to(DEV), y.pin_memory(), grad_W=gW2, chunk_rows=256,
                                             flags=flce.FLCE_FLAG_F32_3PASS)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(a["loss"]) == float(b["loss"]) and torch.equal(a["grad_h"], b["grad_h"]) and torch.equal(gW, gW2)
