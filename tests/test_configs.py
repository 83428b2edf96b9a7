"""Full-size parity on the five LM-head workloads, in the launch configuration
the benchmark times (default chunking, tcgen05 path), against the fp64 oracle.

Every row of the four large heads is compared with the oracle's full forward,
stored under tests/golden/configs by tests/golden/make_config_goldens.py
(which imports only the oracle and the input recipe): the loss within 2e-3
relative, every row's lse, every predicted token (rows whose oracle top-2 gap
is below 1e-3 relative may differ and are counted), and the correct count
exactly, up to those near-tie rows. The inputs are regenerated here from the
same recipe and their sha256 checked against the stored ones first.
Gradients are compared with the oracle run here, one by one: grad_h on 512
seeded rows, and grad_W on 512 vocab rows (the most frequent ids, sampled
labels and a seeded draw) at the head's own N, using every row's lse from the
stored oracle forward. The Llama and Muse heads also run a planted batch: half
of the valid rows relabelled with the oracle's argmax, so that "token accuracy
exact" is tested against an accuracy near 0.5 instead of ~1/V.
Set FLCE_PARITY_REPORT_DIR to write each head's counts there as JSON.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle, oracle_grad_W_rows, oracle_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)
NAMES = ["llama", "muse", "dsv3", "frozen_ce", "frozen_grad_h"]
GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "configs")
GOLDEN_FOR = {"llama": "llama", "muse": "muse", "dsv3": "dsv3", "frozen_ce": "frozen", "frozen_grad_h": "frozen"}


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _golden(name):
    g = GOLDEN_FOR[name]
    with open(os.path.join(GOLDEN_DIR, g + ".json")) as f:
        meta = json.load(f)
    arrays = dict(np.load(os.path.join(GOLDEN_DIR, g + ".npz")))
    return meta, arrays


def _check_inputs(meta, h, W, y):
    got = {"h": workloads.tensor_sha256(h), "W": workloads.tensor_sha256(W), "labels": workloads.tensor_sha256(y)}
    for k, v in got.items():
        assert v == meta["sha256"][k], (
            f"the input recipe drew different {k} here than when the goldens were written "
            f"(torch {torch.__version__} here, {meta['torch']} there): regenerate them, this is not a kernel error")


def _report(name, rec):
    print(f"{name}: " + json.dumps(rec, sort_keys=True))
    d = os.environ.get("FLCE_PARITY_REPORT_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, f"parity_{name}.json"), "w") as f:
            json.dump(rec, f, indent=1, sort_keys=True)


def _compare_forward(pred_gpu, lse_gpu, y, correct_gpu, meta, arrays, oracle_correct, oracle_loss, loss_gpu):
    """Row-by-row comparison of a full forward with the stored oracle forward;
    returns the counts of the report."""
    pred_o = arrays["predicted"].astype(np.int64)
    near = arrays["near_tie"].astype(bool)
    yv = y.numpy()
    valid = yv != -100
    lse_o = arrays["lse"].astype(np.float64)
    lse_err = np.abs(lse_gpu - lse_o).max()
    assert lse_err <= 1e-4 * np.abs(lse_o).max(), lse_err
    mism = pred_gpu != pred_o
    assert not np.any(mism & ~near), np.nonzero(mism & ~near)[0][:10]
    # the correct count differs from the oracle's only through rows whose
    # argmax went the other way on a near tie
    shift = int(np.sum(((pred_gpu == yv).astype(np.int64) - (pred_o == yv).astype(np.int64))[mism & valid]))
    assert correct_gpu == oracle_correct + shift, (correct_gpu, oracle_correct, shift)
    rel = abs(loss_gpu - oracle_loss) / abs(oracle_loss)
    assert rel <= 2e-3, (loss_gpu, oracle_loss)
    return {"rows": int(len(yv)), "loss_gpu": loss_gpu, "loss_oracle": oracle_loss, "loss_rel_err": rel,
            "lse_max_abs_err": float(lse_err), "near_tie_rows": int(near.sum()),
            "predicted_mismatches": int(mism.sum()), "predicted_mismatches_off_near_tie": 0,
            "correct_gpu": int(correct_gpu), "correct_oracle": int(oracle_correct),
            "correct_shift_from_near_ties": shift}


@pytest.mark.parametrize("name", NAMES)
def test_full_size_against_oracle(flce, name):
    w = workloads.WORKLOADS[name]
    meta, arrays = _golden(name)
    h, W, y = workloads.make_inputs(w)
    _check_inputs(meta, h, W, y)
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
        # without the predicted tokens, as the training step calls it: the
        # epilogue then skips the argmax, and the count must still be the
        # forward's (which computes the argmax)
        o = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW, return_predicted=False, **kw)
        loss_b, acc_b, gh = o["loss"], o["token_accuracy"], o["grad_h"]
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(loss_b) == float(f["loss"]) and float(acc_b) == float(f["token_accuracy"])
    if w.row_shape is not None:
        assert f["predicted"].shape == tuple(w.row_shape) and f["lse"].shape == tuple(w.row_shape)
        if gh is not None:
            assert gh.shape == (*w.row_shape, w.hidden)

    h2, y2 = h.reshape(-1, w.hidden), y.reshape(-1)
    n_valid = int((y2 != -100).sum())
    assert n_valid == meta["n_valid"]
    pred = f["predicted"].reshape(-1).cpu().numpy()
    lse = f["lse"].reshape(-1).cpu().double().numpy()
    correct_gpu = round(float(f["token_accuracy"]) * n_valid)
    assert correct_gpu == int(np.sum((pred == y2.numpy()) & (y2.numpy() != -100)))
    rec = _compare_forward(pred, lse, y2, correct_gpu, meta, arrays, meta["correct"], meta["loss"], float(f["loss"]))

    # grad_h on sampled rows, each computed by the oracle from its row alone
    if gh is not None:
        rows = workloads.sample_indices(h2.shape[0], 512, seed=100 + w.seed)
        ref = oracle_rows(h2[rows], W, y2[rows], n_valid, need_grad_h=True, **kw)
        g = gh.reshape(-1, w.hidden)[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
        err = np.abs(g - ref["grad_h"]).max() / np.abs(ref["grad_h"]).max()
        assert err <= 1e-2, err
        rec["grad_h_rows_checked"], rec["grad_h_err_over_max"] = int(len(rows)), float(err)

    # grad_W at the head's own N on sampled vocab rows
    if gW is not None:
        labs = [int(v) for v in y2.numpy() if v != -100][:128]
        ids = workloads.sample_indices(w.vocab, 512 - 32 - 1, seed=200 + w.seed,
                                       must_include=workloads.zipf_head_ids(w.vocab, 32) + labs[:64] + [w.vocab - 1])
        ref = oracle_grad_W_rows(h2, W, y2, ids, arrays["lse"].astype(np.float64), n_valid, **kw)
        got = gW[torch.from_numpy(ids).to(DEV)].double().cpu().numpy()
        err = np.abs(got - ref).max() / np.abs(ref).max()
        assert err <= 1e-2, err
        rec["grad_W_rows_checked"], rec["grad_W_err_over_max"] = int(len(ids)), float(err)

        # without softcap the columns of dL/dW sum to zero over the vocabulary,
        # up to the bf16 rounding of dz (at most 2^-9 of each term; the label term
        # -1/n_valid rounds the same way on every row, so the error does not
        # average out): |sum_j gW_jk| <= 2^-8 |m| / n_valid * sum_{valid i} |h_ik|
        if w.softcap == 0.0:
            col = gW.double().sum(dim=0).abs()
            habs = hd.reshape(-1, w.hidden)[yd.reshape(-1) != -100].double().abs().sum(0)
            bound = 2.0 ** -8 * abs(w.out_mult) / n_valid * habs
            assert torch.all(col <= bound), (col.max().item(), bound.min().item())
    _report(name, rec)


@pytest.mark.parametrize("name", ["llama", "muse"])
def test_planted_accuracy_full_size(flce, name):
    """Half of the valid rows relabelled with the oracle's own argmax: the
    token accuracy is then about 0.5, and the GPU's correct count must equal
    the oracle's, up to rows whose argmax is a near tie."""
    w = workloads.WORKLOADS[name]
    meta, arrays = _golden(name)
    h, W, y = workloads.make_inputs(w)
    _check_inputs(meta, h, W, y)
    pl = meta["planted"]
    yp = workloads.plant_labels(y, arrays["predicted"], pl["frac"], pl["seed"])
    assert workloads.tensor_sha256(yp) == pl["sha256_labels"]
    kw = dict(softcap=w.softcap, out_mult=w.out_mult)
    f = flce.flce_forward(h.to(DEV), W.to(DEV), yp.to(DEV), return_lse=True, **kw)
    loss_c, acc_c = flce.flce_ce_only(h.to(DEV), W.to(DEV), yp.to(DEV), **kw)   # no argmax in its epilogue
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert float(loss_c) == float(f["loss"]) and float(acc_c) == float(f["token_accuracy"])
    n_valid = pl["n_valid"]
    pred = f["predicted"].cpu().numpy()
    correct_gpu = round(float(f["token_accuracy"]) * n_valid)
    assert correct_gpu == int(np.sum((pred == yp.numpy()) & (yp.numpy() != -100)))
    assert pl["correct"] >= 0.5 * n_valid
    rec = _compare_forward(pred, f["lse"].cpu().double().numpy(), yp, correct_gpu, meta, arrays, pl["correct"],
                           pl["loss"], float(f["loss"]))
    _report(name + "_planted", rec)


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
