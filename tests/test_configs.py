"""Full-size parity on the five LM-head workloads, in the launch configuration
the benchmark times (default chunking, tcgen05 path).

At these sizes the fp64 oracle cannot run every output, so the checks are:
  * per-row outputs on a seeded sample of 256 rows, each computed by the oracle
    one by one (lse, predicted token, grad_h row), given the batch's n_valid;
  * properties that hold at any size on the full outputs: the loss equals the
    mean over valid rows of lse_i - s_{i,y_i} (label logits recomputed by a
    plain torch gather-dot), the token accuracy equals the GPU's own argmax
    count, and, without softcap, the columns of the grad_W increment sum to 0;
  * grad_W on sampled vocab rows (the most frequent ids, sampled labels and a
    seeded draw) for the same head at N = 1024 rows, where the oracle's full
    forward is cheap.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle, oracle_grad_W_rows, oracle_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)
NAMES = ["llama", "muse", "dsv3", "frozen_ce", "frozen_grad_h"]


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _cap(z, T):
    return T * torch.tanh(z / T) if T > 0 else z


@pytest.mark.parametrize("name", NAMES)
def test_full_size_sampled_rows(flce, name):
    w = workloads.WORKLOADS[name]
    h, W, y = workloads.make_inputs(w)
    if w.row_shape is not None:                     # the DSpine proposal rows [B, k, S, H]
        h = h.view(*w.row_shape, w.hidden)
        y = y.view(*w.row_shape)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    kw = dict(softcap=w.softcap, out_mult=w.out_mult)
    f = flce.flce_forward(hd, Wd, yd, return_lse=True, **kw)
    gW = None
    if w.mode == "ce_only":
        loss_b, acc_b = flce.flce_ce_only(hd, Wd, yd, **kw)
        gh = None
    else:
        gW = torch.zeros(W.shape, dtype=torch.float32, device=DEV) if w.mode == "fwd_bwd" else None
        o = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW, return_predicted=True, **kw)
        loss_b, acc_b, gh = o["loss"], o["token_accuracy"], o["grad_h"]
        assert torch.equal(o["predicted"], f["predicted"])
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(loss_b) == float(f["loss"]) and float(acc_b) == float(f["token_accuracy"])
    if w.row_shape is not None:
        assert f["predicted"].shape == tuple(w.row_shape) and f["lse"].shape == tuple(w.row_shape)
        if gh is not None:
            assert gh.shape == (*w.row_shape, w.hidden)

    h2, y2 = h.reshape(-1, w.hidden), y.reshape(-1)
    yd2 = yd.reshape(-1)
    valid = yd2 != -100
    n_valid = int(valid.sum())
    lse = f["lse"].reshape(-1)
    pred = f["predicted"].reshape(-1)

    # property: loss = mean over valid rows of lse_i - s_{i, y_i}
    yi = yd2.clamp(min=0)
    z_lab = (hd.reshape(-1, w.hidden).float() * Wd[yi].float()).sum(1) * w.out_mult
    s_lab = _cap(z_lab, w.softcap)
    loss_prop = ((lse.double() - s_lab.double())[valid]).sum().item() / n_valid
    assert abs(float(f["loss"]) - loss_prop) <= 1e-4 * abs(loss_prop), (float(f["loss"]), loss_prop)
    # property: accuracy = the GPU's own argmax count
    assert round(float(f["token_accuracy"]) * n_valid) == int(((pred == yd2) & valid).sum())

    # per-row outputs on a seeded sample of rows, oracle one by one
    rows = workloads.sample_indices(h2.shape[0], 256, seed=100 + w.seed)
    ref = oracle_rows(h2[rows], W, y2[rows], n_valid, need_grad_h=gh is not None, **kw)
    l_gpu = lse.cpu().double().numpy()[rows]
    assert np.abs(l_gpu - ref["lse"]).max() <= 1e-4 * np.abs(ref["lse"]).max()
    p_gpu = pred.cpu().numpy()[rows]
    near = ref["top2_gap"] < 1e-3
    assert np.all((p_gpu == ref["predicted"]) | near), np.nonzero((p_gpu != ref["predicted"]) & ~near)
    print(f"{name}: {int(near.sum())} near-tie rows of {len(rows)} sampled")
    if gh is not None:
        g = gh.reshape(-1, w.hidden)[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
        scale = np.abs(ref["grad_h"]).max()
        assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * scale

    # property: without softcap the columns of dL/dW sum to zero over the vocabulary,
    # up to the bf16 rounding of dz (at most 2^-9 of each term; the label term
    # -1/n_valid rounds the same way on every row, so the error does not average
    # out): |sum_j gW_jk| <= 2^-8 |m| / n_valid * sum_{valid i} |h_ik|
    if gW is not None and w.softcap == 0.0:
        col = gW.double().sum(dim=0).abs()
        habs = hd.reshape(-1, w.hidden)[valid].double().abs().sum(0)
        bound = 2.0 ** -8 * abs(w.out_mult) / n_valid * habs
        assert torch.all(col <= bound), (col.max().item(), bound.min().item())
        # a lost or doubled chunk would leave sums of the order of sum_i h_ik / n_valid
        print(f"{name}: max column sum {col.max().item():.3e}, bound {bound.min().item():.3e}")


@pytest.mark.parametrize("name", ["llama", "muse", "dsv3"])
def test_grad_W_sampled_vocab_rows_full_head(flce, name):
    w = workloads.WORKLOADS[name]
    N = 1024
    h, W, y = workloads.make_inputs(w, n_rows=N)
    kw = dict(softcap=w.softcap, out_mult=w.out_mult)
    gW = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    o = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, **kw)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    full = flce_oracle(h, W, y, need_grad_h=True, need_grad_W=False, **kw)
    assert abs(float(o["loss"]) - full["loss"]) <= 2e-3 * abs(full["loss"])
    gh = o["grad_h"].float().cpu().numpy()
    assert np.abs(gh - full["grad_h"]).max() <= 1e-2 * np.abs(full["grad_h"]).max()
    labs = [int(v) for v in y.numpy() if v != -100][:64]
    ids = workloads.sample_indices(w.vocab, 192, seed=200 + w.seed,
                                   must_include=workloads.zipf_head_ids(w.vocab, 32) + labs + [w.vocab - 1])
    ref = oracle_grad_W_rows(h, W, y, ids, full["lse"], full["n_valid"], **kw)
    got = gW[torch.from_numpy(ids).to(DEV)].double().cpu().numpy()
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


def test_largest_chunk_matches_default_chunking(flce):
    """The largest chunk (32768 rows) on the DSV3 head: its logits buffer holds
    32768 x 129280 = 4.2e9 elements, past 32-bit indexing, and one chunk replaces
    four. Per-row results do not depend on the chunking, so lse, the predicted
    tokens and grad_h must equal the default (8192-row) run's bit for bit; the
    loss differs only by the grouping of its fp64 chunk sums, and grad_W by the
    order of its fp32 chunk additions. Those sums cancel heavily on the Zipf head
    ids (partial sums far larger than the result), so the bound on grad_W is
    1e-4 of its largest entry (measured 2.5e-5): a lost or doubled chunk would
    be off by the order of the entries themselves."""
    w = workloads.WORKLOADS["dsv3"]
    h, W, y = workloads.make_inputs(w)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    runs = []
    for chunk in (0, 32768):
        gW = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
        o = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW, return_predicted=True, chunk_rows=chunk)
        f = flce.flce_forward(hd, Wd, yd, return_lse=True, chunk_rows=chunk)
        torch.cuda.synchronize()
        assert flce.flce_get_status() == 0
        runs.append((o, f, gW))
        flce._workspaces.clear()
        torch.cuda.empty_cache()
    (o1, f1, g1), (o2, f2, g2) = runs
    assert torch.equal(o1["predicted"], o2["predicted"]) and torch.equal(f1["lse"], f2["lse"])
    assert torch.equal(o1["grad_h"], o2["grad_h"])
    assert float(o1["token_accuracy"]) == float(o2["token_accuracy"])
    assert abs(float(o1["loss"]) - float(o2["loss"])) <= 1e-6 * abs(float(o1["loss"]))
    d = (g1 - g2).abs().max().item()
    assert d <= 1e-4 * g1.abs().max().item(), d


@pytest.fixture(scope="module")
def dsv3_inputs():
    w = workloads.WORKLOADS["dsv3"]
    h, W, y = workloads.make_inputs(w)
    return w, h, W, y


def _fwd_bwd(flce, hd, Wd, yd, **kw):
    gW = torch.zeros(Wd.shape, dtype=torch.float32, device=DEV)
    o = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW, return_predicted=True, **kw)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    flce.flce_release_workspaces()
    return o


def test_tile_shapes_agree_bit_for_bit_full_head(flce, dsv3_inputs):
    """The DSV3 head in the benchmark's configuration on 256 x 256 tiles (the
    default) and on 128 x 256 tiles: each output element is accumulated over
    the same K order either way, so every output agrees bit for bit."""
    w, h, W, y = dsv3_inputs
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    a = _fwd_bwd(flce, hd, Wd, yd)
    b = _fwd_bwd(flce, hd, Wd, yd, flags=flce.FLCE_FLAG_TILE128)
    assert float(a["loss"]) == float(b["loss"]) and float(a["token_accuracy"]) == float(b["token_accuracy"])
    for k in ("predicted", "grad_h", "grad_W"):
        assert torch.equal(a[k], b[k]), k


def test_low_memory_backward_matches_stored_logits_full_head(flce, dsv3_inputs):
    """The recompute backward on the full DSV3 head: the forward is the same
    kernel, so loss, accuracy and predictions are equal; the gradients differ
    only by how dlogits' exponential is evaluated before the bf16 rounding."""
    w, h, W, y = dsv3_inputs
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    a = _fwd_bwd(flce, hd, Wd, yd)
    b = _fwd_bwd(flce, hd, Wd, yd, low_memory=True)
    assert float(a["loss"]) == float(b["loss"]) and float(a["token_accuracy"]) == float(b["token_accuracy"])
    assert torch.equal(a["predicted"], b["predicted"])
    # grad_h is bf16: one rounding flip of its largest entries is 2^-8 of them;
    # grad_W (fp32) differs by the few dz entries whose bf16 rounding flipped
    for k, tol in (("grad_h", 2.0 ** -7), ("grad_W", 1e-3)):
        x, z = a[k].float(), b[k].float()
        assert (x - z).abs().max().item() <= tol * x.abs().max().item(), k


def test_fp32_inputs_full_size_sampled_rows(flce, dsv3_inputs):
    """The tf32 path on the full DSV3 head (fp32 h and W holding the bf16
    values): per-row lse, predicted token and grad_h on sampled rows against
    the oracle one by one, and the loss against the bf16 path's."""
    w, h, W, y = dsv3_inputs
    hd, Wd, yd = h.float().to(DEV), W.float().to(DEV), y.to(DEV)
    o = flce.flce_forward_backward(hd, Wd, yd, return_predicted=True)
    f = flce.flce_forward(hd, Wd, yd, return_lse=True)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    n_valid = int((y != -100).sum())
    rows = workloads.sample_indices(w.n_rows, 128, seed=300)
    ref = oracle_rows(h[rows], W, y[rows], n_valid)
    lse = f["lse"].cpu().double().numpy()[rows]
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * np.abs(ref["lse"]).max()
    pred = o["predicted"].cpu().numpy()[rows]
    assert np.all((pred == ref["predicted"]) | (ref["top2_gap"] < 1e-3))
    g = o["grad_h"][torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * np.abs(ref["grad_h"]).max()
    flce.flce_release_workspaces()
    b = _fwd_bwd(flce, h.to(DEV), W.to(DEV), yd)
    assert abs(float(o["loss"]) - float(b["loss"])) <= 2e-3 * abs(float(b["loss"]))


def test_repeated_calls_are_bit_reproducible(flce, dsv3_inputs):
    """Twenty forward+backward calls on the DSV3 head, on two streams in turn:
    the merge sums in a fixed order and no kernel uses atomics for its results,
    so the loss, accuracy, predictions and grad_h are the same bits every time,
    and every call leaves the device status at 0."""
    w, h, W, y = dsv3_inputs
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    streams = [torch.cuda.current_stream(DEV), torch.cuda.Stream(DEV)]
    first = None
    for it in range(20):
        s = streams[it % 2]
        s.wait_stream(torch.cuda.current_stream(DEV))
        with torch.cuda.stream(s):
            o = flce.flce_forward_backward(hd, Wd, yd, return_predicted=True)
            s.synchronize()
            assert flce.flce_get_status() == 0, it
        if first is None:
            first = o
            continue
        assert float(o["loss"]) == float(first["loss"]) and float(o["token_accuracy"]) == float(
            first["token_accuracy"]), it
        assert torch.equal(o["predicted"], first["predicted"]) and torch.equal(o["grad_h"], first["grad_h"]), it
    flce.flce_release_workspaces()
