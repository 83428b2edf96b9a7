"""The softcap's polynomial form, pinned on the CPU.

Where every |u / T| of a warp's 32-column group is below 1/2, the epilogues
compute s = T tanh(u / T) as u P((u / T)^2), with P of degree 5 (constant term
1) fitted by least squares on 4000 Chebyshev nodes of [0, 1/4] to tanh(x) / x.
These tests read the coefficients out of the CUDA source, re-derive them from
that definition, evaluate the form as the kernel does (fp32, correctly rounded
FMAs, the same operation order) and bound its error against fp64 tanh.
"""
import os
import re

import numpy as np
import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "linear_cross_entropy_02_gb300", "csrc", "flce_epilogue.cuh")


def _source_coefficients():
    text = open(SRC).read()
    body = text[text.index("void softcap32("):]
    body = body[:body.index("float xmax")]
    vals = {}
    for name, a, b in re.findall(r"const uint64_t (p\d) = f2_pack\(([-0-9.e]+)f, ([-0-9.e]+)f\);", body):
        assert a == b
        vals[int(name[1:])] = float(a)
    assert sorted(vals) == [0, 1, 2, 3, 4, 5]
    return np.array([vals[k] for k in range(6)], dtype=np.float32)


def _fit(deg=5, n=4000, w_max=0.25):
    k = np.arange(n)
    w = w_max * (1 - np.cos(np.pi * (k + 0.5) / n)) / 2
    x = np.sqrt(w)
    f = np.tanh(x) / x
    A = np.vander(w, deg, increasing=True)
    c, *_ = np.linalg.lstsq(A, (f - 1) / w, rcond=None)
    return np.concatenate([[1.0], c])


def _f32(a):
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def _kernel_form(u, T, c):
    """u P((u/T)^2) in the kernel's order: x = u * (1/T), w = x * x, Horner by FMA, s = u * q."""
    inv_t = np.float32(1.0 / np.float32(T))
    x = _f32(u.astype(np.float64) * np.float64(inv_t))
    w = _f32(x.astype(np.float64) * x.astype(np.float64))
    q = np.full_like(w, c[5])
    for k in (4, 3, 2, 1, 0):
        q = _f32(q.astype(np.float64) * w.astype(np.float64) + np.float64(c[k]))
    return _f32(u.astype(np.float64) * q.astype(np.float64))


def test_coefficients_are_the_stated_fit():
    c = _source_coefficients()
    fit = _f32(_fit())
    assert c[0] == 1.0
    ulps = np.abs(c.astype(np.float64) - fit.astype(np.float64)) / np.spacing(np.abs(fit))
    assert np.all(ulps <= 1.0), (c, fit)


def test_coefficients_follow_the_power_series_of_tanh():
    # tanh(x)/x = 1 - w/3 + 2w^2/15 - 17w^3/315 + 62w^4/2835 - ..., w = x^2: a fit on a
    # small interval lands near the leading terms (a sign or index slip would not)
    c = _source_coefficients().astype(np.float64)
    assert abs(c[1] + 1 / 3) < 1e-6
    assert abs(c[2] - 2 / 15) < 1e-5
    assert abs(c[3] + 17 / 315) < 1e-3
    assert abs(c[4] - 62 / 2835) < 1e-3


def test_error_bound_against_fp64_tanh():
    c = _source_coefficients()
    for T in (1.0, 2.5, 30.0, 100.0):
        u = np.linspace(-0.4999 * T, 0.4999 * T, 400001).astype(np.float32)
        s = _kernel_form(u, T, c)
        ref = np.float64(np.float32(T)) * np.tanh(u.astype(np.float64) / np.float64(np.float32(T)))
        nz = ref != 0
        ulp = np.abs(s[nz] - ref[nz]) / np.spacing(np.abs(ref[nz]).astype(np.float32)).astype(np.float64)
        assert ulp.max() <= 1.2, (T, ulp.max())
        # odd, and exact at 0 with its sign
        assert np.array_equal(_kernel_form(-u, T, c), -s)
    z = _kernel_form(np.array([0.0, -0.0], dtype=np.float32), 30.0, c)
    assert z[0] == 0 and not np.signbit(z[0]) and np.signbit(z[1])


@pytest.mark.gpu
@pytest.mark.parametrize("softcap", [0.5, 5.5, 30.0])
def test_capped_row_lse_against_fp64(softcap):
    """Every row's lse on the GPU against the fp64 oracle, to 2e-6 relative.
    The logits z have a standard deviation of 0.8: with T = 30 every 32 x 32
    group of a warp takes the polynomial form, with T = 0.5 every group falls
    back to tanhf, and with T = 5.5 (|z| > T/2 at 3.4 sigma) about half the
    groups take each, within the same rows."""
    import torch

    import __graft_entry__
    import workloads
    from oracle import flce_oracle
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as flce

    N, H, V = 256, 256, 3000
    h = workloads.make_hidden(N, H, 61)
    W = workloads.make_weight(V, H, 61, std=0.1)
    y = workloads.make_labels(N, V, 61, 0.1)
    dev = torch.device("cuda", 0)
    f = flce.flce_forward(h.to(dev), W.to(dev), y.to(dev), softcap=softcap, out_mult=0.5, return_lse=True)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, softcap=softcap, out_mult=0.5, need_grad_h=False, need_grad_W=False)
    lse = f["lse"].double().cpu().numpy()
    rel = np.abs(lse - ref["lse"]) / np.abs(ref["lse"])
    assert rel.max() <= 2e-6, rel.max()
