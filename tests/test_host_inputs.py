"""flce_forward_backward_from_host and flce_ce_only_from_host: h and labels in
host memory, copied chunk by chunk by the library under its own kernels. The kernels and their inputs are the
same as with device inputs, so every output must equal the device-input call's
bit for bit; the parity of that call with the oracle is covered elsewhere, and
one case here also goes to the oracle directly."""
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


def _same(a, b):
    return (a is None and b is None) or torch.equal(a.cpu(), b.cpu())


def _both(flce, h, W, y, **kw):
    """The host-input call and the device-input call on the same data."""
    V, H = W.shape
    gW1 = torch.full((V, H), 0.125, dtype=torch.float32, device=DEV)
    gW2 = gW1.clone()
    o1 = flce.flce_forward_backward_from_host(h, W.to(DEV), y, grad_W=gW1, return_predicted=True, **kw)
    o2 = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW2, return_predicted=True, **kw)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    return o1, o2


@pytest.mark.parametrize("case", [
    dict(N=300, H=192, V=1000, chunk_rows=128),                # 3 chunks, ragged last chunk
    dict(N=1000, H=256, V=3000, chunk_rows=128, softcap=30.0, out_mult=0.5),   # 8 chunks: buffers reused
    dict(N=513, H=136, V=777, chunk_rows=256, low_memory=True, vocab_slab=256),
    dict(N=64, H=64, V=500),                                   # one chunk
])
def test_host_inputs_equal_device_inputs(flce, case):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h = workloads.make_hidden(N, H, N + V).pin_memory()
    W = workloads.make_weight(V, H, N + V, std=0.05)
    y = workloads.make_labels(N, V, N + V, 0.1).pin_memory()
    o1, o2 = _both(flce, h, W, y, **c)
    assert float(o1["loss"]) == float(o2["loss"]) and float(o1["token_accuracy"]) == float(o2["token_accuracy"])
    for k in ("predicted", "grad_h", "grad_W"):
        assert _same(o1[k], o2[k]), k
    assert o1["loss"].device.type == "cpu" and o1["grad_h"].device.type == "cuda"


def test_host_inputs_strided_pageable_and_back_to_back(flce):
    """Rows of h with a stride wider than H, from pageable (not page-locked)
    memory; then three calls queued back to back on one stream with different
    inputs, which reuse the same staging buffers."""
    N, H, V = 400, 128, 2000
    wide = workloads.make_hidden(N, H + 64, 5)
    h = wide[:, :H]                                     # ld_h = H + 64
    W = workloads.make_weight(V, H, 5, std=0.05)
    y = workloads.make_labels(N, V, 5, 0.1)
    o1, o2 = _both(flce, h, W, y, chunk_rows=128)
    assert float(o1["loss"]) == float(o2["loss"]) and _same(o1["grad_h"], o2["grad_h"])
    ref = flce_oracle(h, W, y)
    check_against_oracle({k: o1[k] for k in ("loss", "token_accuracy", "predicted", "grad_h")}, ref, y,
                         what="host inputs")

    hs = [workloads.make_hidden(N, H, 10 + i).pin_memory() for i in range(3)]
    ys = [workloads.make_labels(N, V, 10 + i, 0.1).pin_memory() for i in range(3)]
    Wd = W.to(DEV)
    outs = [flce.flce_forward_backward_from_host(hs[i], Wd, ys[i], chunk_rows=128) for i in range(3)]
    torch.cuda.synchronize()
    for i in range(3):
        r = flce.flce_forward_backward(hs[i].to(DEV), Wd, ys[i].to(DEV), chunk_rows=128)
        torch.cuda.synchronize()
        assert float(outs[i]["loss"]) == float(r["loss"]), i
        assert torch.equal(outs[i]["grad_h"], r["grad_h"]), i


def test_ce_only_from_host_equals_device_inputs(flce):
    N, H, V = 1000, 256, 3000
    h = workloads.make_hidden(N, H, 31).view(4, 250, H).pin_memory()   # leading dims are flattened
    W = workloads.make_weight(V, H, 31, std=0.05).to(DEV)
    y = workloads.make_labels(N, V, 31, 0.1).view(4, 250).pin_memory()
    l1, a1 = flce.flce_ce_only_from_host(h, W, y, softcap=30.0, chunk_rows=128)
    l2, a2 = flce.flce_ce_only(h.to(DEV), W, y.to(DEV), softcap=30.0, chunk_rows=128)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(l1) == float(l2) and float(a1) == float(a2)


@pytest.mark.parametrize("flags", [0, 32])
def test_fp32_host_inputs_equal_device_inputs(flce, flags):
    """The tf32 path from host buffers: fp32 h staged with 4-byte rows."""
    N, H, V = 500, 136, 1000
    g = torch.Generator().manual_seed(9)
    h = torch.randn((N, H), generator=g).pin_memory()
    W = torch.randn((V, H), generator=g) * 0.05
    y = workloads.make_labels(N, V, 9, 0.1).pin_memory()
    Wd = W.to(DEV)
    gW1 = torch.zeros((V, H), device=DEV)
    gW2 = torch.zeros((V, H), device=DEV)
    o1 = flce.flce_forward_backward_from_host(h, Wd, y, grad_W=gW1, return_predicted=True, chunk_rows=128,
                                              flags=flags)
    o2 = flce.flce_forward_backward(h.to(DEV), Wd, y.to(DEV), grad_W=gW2, return_predicted=True, chunk_rows=128,
                                    flags=flags)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(o1["loss"]) == float(o2["loss"]) and o1["grad_h"].dtype == torch.float32
    for k in ("predicted", "grad_h", "grad_W"):
        assert _same(o1[k], o2[k]), k
    l1, a1 = flce.flce_ce_only_from_host(h, Wd, y, chunk_rows=128)
    torch.cuda.synchronize()
    assert float(l1) == float(o2["loss"])


def test_host_inputs_rejections(flce):
    h = workloads.make_hidden(16, 64, 1)
    W = workloads.make_weight(100, 64, 1).to(DEV)
    y = workloads.make_labels(16, 100, 1, 0.0)
    with pytest.raises(ValueError):
        flce.flce_forward_backward_from_host(h.to(DEV), W, y)            # h must be on the host
    with pytest.raises(ValueError):
        flce.flce_forward_backward_from_host(h.float(), W, y)            # dtypes must match
    with pytest.raises(flce.FlceError):
        flce.flce_forward_backward_from_host(h, W, y, flags=flce.FLCE_FLAG_SIMT_GEMM)
    np.testing.assert_equal(flce.flce_get_status(), 0)
