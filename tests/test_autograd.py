"""The differentiable form of the fused head (autograd function and module) and
the gradient-scaling kernel it uses, on the GPU, against the fp64 oracle. The
pages use the fused loss inside a model's forward and let autograd carry the
gradients on (DeepSeek-V3 page, Summary; Muse Glimmer page, Summary item 1);
a frozen projection gets no weight gradient (SpecForge DSpine PR, Changes)."""
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


def _inputs(N, H, V, seed, ign=0.1):
    h = workloads.make_hidden(N, H, seed)
    W = workloads.make_weight(V, H, seed)
    y = workloads.make_labels(N, V, seed, ign)
    return h, W, y


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 4096, 100003])
@pytest.mark.parametrize("pair", [("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16"), ("bf16", "f32")])
def test_scale_gradient_matches_torch_bitwise(flce, n, pair):
    """y = s * x rounded to y's type: fp32 product, then round to nearest even,
    which is what torch's (x.float() * s).to(dtype) computes, so the two agree
    bit for bit; aligned and misaligned (offset by one element) arrays."""
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}
    g = torch.Generator().manual_seed(n + 17)
    base = (torch.randn(n + 1, generator=g) * 3.0).to(dt[pair[0]]).to(DEV)
    s = torch.tensor([0.7371], dtype=torch.float32, device=DEV)
    for x in (base[:n], base[1:]):
        y = flce.flce_scale_gradient(x, s, out_dtype=dt[pair[1]])
        ref = (x.float() * s).to(dt[pair[1]])
        assert torch.equal(y.view(-1), ref.view(-1))
    y1 = flce.flce_scale_gradient(base, None, out_dtype=dt[pair[1]])
    assert torch.equal(y1, base.to(dt[pair[1]]))


def test_scale_gradient_in_place(flce):
    x = torch.randn(1 << 20, device=DEV)
    ref = x * 0.25
    out = flce.flce_scale_gradient(x, torch.tensor([0.25], device=DEV), out=x)
    assert out.data_ptr() == x.data_ptr() and torch.equal(x, ref)
    with pytest.raises(ValueError):
        flce.flce_scale_gradient(x, torch.tensor([0.25], device=DEV), out=x, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("case", [
    dict(N=256, H=512, V=4096),
    dict(N=300, H=192, V=1000, chunk_rows=128, softcap=30.0, out_mult=0.5),
    dict(N=129, H=64, V=4100, reduction="sum"),
])
def test_autograd_grads_match_oracle(flce, case):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h, W, y = _inputs(N, H, V, seed=N + V)
    hd = h.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    loss, acc = flce.linear_cross_entropy(hd, Wd, y.to(DEV), **c)
    assert loss.requires_grad and not acc.requires_grad
    loss.backward()
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert hd.grad.dtype == torch.bfloat16 and Wd.grad.dtype == torch.bfloat16
    ref = flce_oracle(h, W, y, softcap=c.get("softcap", 0.0), out_mult=c.get("out_mult", 1.0),
                      reduction=c.get("reduction", "mean"))
    out = {"loss": loss.detach(), "token_accuracy": acc, "grad_h": hd.grad}
    check_against_oracle(out, ref, y, what=f"autograd {case}")
    # W's gradient reaches autograd in W's dtype: compare the bf16 values with
    # the oracle's grad_W at the grad tolerance plus one bf16 rounding
    gW = Wd.grad.double().cpu().numpy()
    scale = np.abs(ref["grad_W"]).max()
    assert np.abs(gW - ref["grad_W"]).max() <= 1e-2 * scale + 2.0 ** -8 * np.abs(ref["grad_W"]).max()


def test_autograd_upstream_factor(flce):
    """d(k * loss)/d(inputs) = k * grads. For k = 2 (a power of two) the
    gradient equals, bit for bit, the fused call with grad_scale = 2: scaling
    by 2 commutes with every rounding on the way. For k = 0.3 it matches the
    oracle run with grad_scale 0.3."""
    N, H, V = 256, 256, 3000
    h, W, y = _inputs(N, H, V, seed=5)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    ref2 = flce.flce_forward_backward(hd, Wd, yd, grad_W=torch.zeros(V, H, device=DEV), grad_scale=2.0)
    a = hd.clone().requires_grad_(True)
    b = Wd.float().clone().requires_grad_(True)   # fp32 W: the fp32 accumulator reaches .grad unrounded
    loss, _ = flce.linear_cross_entropy(a, b.bfloat16(), yd)
    (2.0 * loss).backward()
    torch.cuda.synchronize()
    assert torch.equal(a.grad, ref2["grad_h"])
    # b.bfloat16() is a cast node: autograd hands the bf16 gradient back through it
    assert torch.equal(b.grad, ref2["grad_W"].bfloat16().float())

    c = hd.clone().requires_grad_(True)
    loss, acc = flce.linear_cross_entropy(c, Wd, yd)
    (0.3 * loss).backward()
    torch.cuda.synchronize()
    ref = flce_oracle(h, W, y, grad_scale=0.3, need_grad_W=False)
    check_against_oracle({"loss": loss.detach(), "token_accuracy": acc, "grad_h": c.grad}, ref, y,
                         what="upstream 0.3")


def test_autograd_frozen_weight_and_module(flce):
    """A frozen W (requires_grad False) gets no gradient and costs no grad_W
    GEMM; the module form returns the same loss as the function."""
    N, H, V = 512, 256, 5000
    h, W, y = _inputs(N, H, V, seed=11)
    hd = h.to(DEV).requires_grad_(True)
    Wd = W.to(DEV)
    mod = flce.FusedLinearCrossEntropyLoss(softcap=30.0, return_token_accuracy=True)
    flce.flce_profile_begin(True)
    loss, acc = mod(hd.view(2, 256, H), Wd, y.to(DEV).view(2, 256))
    loss.backward()
    kernels = flce.flce_profile_read()
    flce.flce_profile_begin(False)
    torch.cuda.synchronize()
    assert "grad_W_gemm" not in kernels and "grad_h_gemm" in kernels
    assert Wd.grad is None and hd.grad.shape == (N, H)
    ref = flce_oracle(h, W, y, softcap=30.0, need_grad_W=False)
    check_against_oracle({"loss": loss.detach(), "token_accuracy": acc, "grad_h": hd.grad}, ref, y,
                         what="frozen module")
    with torch.no_grad():
        l2 = flce.FusedLinearCrossEntropyLoss(softcap=30.0)(hd.detach(), Wd, y.to(DEV))
    assert float(l2) == float(loss)


def test_autograd_on_256_row_tiles(flce):
    """The same autograd gradients through the 256-row GEMM tiles (forced: at
    this size each GEMM would otherwise pick 128-row tiles)."""
    N, H, V = 300, 192, 1000
    h, W, y = _inputs(N, H, V, seed=21)
    hd = h.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    loss, acc = flce.linear_cross_entropy(hd, Wd, y.to(DEV), softcap=30.0, out_mult=0.5, chunk_rows=128)
    loss.backward()
    ref_loss, ref_acc = float(loss), float(acc)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=torch.zeros(V, H, device=DEV),
                                     softcap=30.0, out_mult=0.5, chunk_rows=128, flags=flce.FLCE_FLAG_TILE256)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, softcap=30.0, out_mult=0.5)
    check_against_oracle(out, ref, y, what="tile256")
    check_against_oracle({"loss": loss.detach(), "token_accuracy": acc, "grad_h": hd.grad}, ref, y,
                         what="autograd default tiles")
    assert abs(float(out["loss"]) - ref_loss) <= 1e-6 * abs(ref_loss) and float(out["token_accuracy"]) == ref_acc


def test_autograd_rejects_per_row_reduction(flce):
    h, W, y = _inputs(16, 64, 100, seed=3)
    with pytest.raises(ValueError):
        flce.linear_cross_entropy(h.to(DEV), W.to(DEV), y.to(DEV), reduction="none")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("need_gh", [True, False])
def test_second_backward_through_the_node_raises(flce, dtype, need_gh):
    """The backward scales the saved gradients in place (grad_h, and an fp32
    grad_W); a second backward through the same node (retain_graph=True) would
    scale them twice, so it must fail loudly with autograd's in-place error.
    With bf16 W and no grad_h nothing saved is modified, and a second backward
    gives the same gradient again."""
    N, H, V = 128, 64, 500
    h, W, y = _inputs(N, H, V, seed=31)
    hd = h.to(DEV).to(dtype).requires_grad_(need_gh)
    Wd = W.to(DEV).to(dtype).requires_grad_(True)
    loss, _ = flce.linear_cross_entropy(hd, Wd, y.to(DEV))
    (3.0 * loss).backward(retain_graph=True)
    if not need_gh:
        gW1 = Wd.grad.clone()
        if dtype == torch.bfloat16:
            Wd.grad = None
            (3.0 * loss).backward()
            assert torch.equal(Wd.grad, gW1)
        else:
            with pytest.raises(RuntimeError, match="inplace"):
                loss.backward()
            assert torch.equal(Wd.grad, gW1)
        return
    g1 = hd.grad.clone()
    with pytest.raises(RuntimeError, match="inplace"):
        loss.backward()
    torch.cuda.synchronize()
    assert torch.equal(hd.grad, g1)                  # the failed backward left the gradient as it was
