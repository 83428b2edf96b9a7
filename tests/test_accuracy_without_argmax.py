"""Token accuracy on calls that return no predicted tokens.

Such calls (CE-only, and the forward or forward+backward without
`return_predicted`) skip the argmax in the forward GEMM's epilogue: each
256-column vocab tile records only whether the row's label is the tile's first
maximum, and the merge takes the first tile that holds the row's maximum, as it
does for the argmax. These tests pin that the correct count, the loss and the
gradients are those of the argmax path bit for bit, on planted exact ties at
every level of the walk (within a 32-column group, across groups of a tile,
across tiles that different merge warps fold, at tile edges, in the masked last
tile), on every GEMM path, and against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _count(acc, y):
    n_valid = int((y != -100).sum())
    return round(float(acc) * n_valid)


def _all_paths(flce, h, W, y, flags=0, **kw):
    """The correct count, loss and gradients from every entry point, with and
    without the predicted tokens."""
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    gW1 = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    gW2 = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    a = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW1, return_predicted=True, flags=flags, **kw)
    b = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW2, return_predicted=False, flags=flags, **kw)
    f1 = flce.flce_forward(hd, Wd, yd, return_predicted=True, flags=flags, **kw)
    f2 = flce.flce_forward(hd, Wd, yd, return_predicted=False, return_lse=True, flags=flags, **kw)
    loss_c, acc_c = flce.flce_ce_only(hd, Wd, yd, flags=flags, **kw)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert b["predicted"] is None and f2["predicted"] is None
    counts = {k: _count(v, y) for k, v in (("fb_pred", a["token_accuracy"]), ("fb", b["token_accuracy"]),
                                            ("fwd_pred", f1["token_accuracy"]), ("fwd", f2["token_accuracy"]),
                                            ("ce", acc_c))}
    losses = {float(a["loss"]), float(b["loss"]), float(f1["loss"]), float(f2["loss"]), float(loss_c)}
    assert len(losses) == 1, losses
    assert torch.equal(a["grad_h"], b["grad_h"]) and torch.equal(gW1, gW2)
    pred = a["predicted"].cpu()
    assert torch.equal(pred, f1["predicted"].cpu())
    valid = y != -100
    from_pred = int(((pred == y) & valid).sum())
    return counts, from_pred, pred


def _tie_inputs(N, H, V, cols, seed):
    """Rows of W at `cols` set to one identical dominating vector (and every
    row of h positive), so those columns tie bit for bit at every row's max."""
    h = workloads.make_hidden(N, H, seed).abs()
    W = workloads.make_weight(V, H, seed)
    for c in cols:
        W[c] = 0.5
    return h, W


# column sets that tie: within one 32-column group, across groups of one
# 256-column tile, across tiles folded by different merge warps, at the two
# sides of a tile edge, and in the last (masked) tile of V = 1500
TIES = [
    ("group", [64 + 3, 64 + 8]),
    ("group_three", [96, 97, 127]),
    ("tile_groups", [256 + 10, 256 + 100]),
    ("tiles", [300, 1210]),
    ("tile_edge", [255, 256]),
    ("tile_edge_first_col", [512, 700]),
    ("tile_second_group", [520, 700]),
    ("last_tile", [1280, 1499]),
]


@pytest.mark.parametrize("flags_name", ["default", "tile128", "tile256"])
@pytest.mark.parametrize("tie_name,cols", TIES, ids=[t[0] for t in TIES])
def test_planted_exact_ties(flce, tie_name, cols, flags_name):
    flags = {"default": 0, "tile128": flce.FLCE_FLAG_TILE128, "tile256": flce.FLCE_FLAG_TILE256}[flags_name]
    N, H, V = 96, 128, 1500
    h, W = _tie_inputs(N, H, V, cols, seed=41)
    y = workloads.make_labels(N, V, 41, 0.1)
    # label every tied column on some rows: only the lowest one is the argmax
    for i, c in enumerate(cols):
        y[10 * i:10 * i + 10] = c
    y[40:45] = cols[0] + 1 if cols[0] + 1 not in cols else cols[0] - 1   # beside the first maximum
    start = (cols[0] // 256) * 256
    if start not in cols:
        y[45:50] = start      # the first column of the maximum's tile, not itself a maximum
    counts, from_pred, pred = _all_paths(flce, h, W, y, flags=flags)
    assert torch.all(pred == min(cols))
    expect = int(((y == min(cols)) & (y != -100)).sum())
    assert from_pred == expect >= 10
    assert set(counts.values()) == {expect}, counts


@pytest.mark.parametrize("flags_name", ["default", "tile128", "tile256", "kmajor", "recompute", "simt"])
@pytest.mark.parametrize("softcap,out_mult", [(0.0, 1.0), (30.0, 0.5), (0.0, 0.5)])
def test_planted_accuracy_matches_argmax_path_and_oracle(flce, flags_name, softcap, out_mult):
    """A third of the valid rows labelled with the row's own argmax, on a ragged
    head (several row and vocab tiles, masked tails): every entry point gives
    the same correct count, and it is the oracle's off its near-tie rows."""
    flags = {"default": 0, "tile128": flce.FLCE_FLAG_TILE128, "tile256": flce.FLCE_FLAG_TILE256,
             "kmajor": flce.FLCE_FLAG_KMAJOR_BWD, "recompute": flce.FLCE_FLAG_RECOMPUTE,
             "simt": flce.FLCE_FLAG_SIMT_GEMM}[flags_name]
    N, H, V = 300, 192, 4099
    h = workloads.make_hidden(N, H, 42)
    W = workloads.make_weight(V, H, 42, std=0.1)
    y = workloads.make_labels(N, V, 42, 0.1)
    ref = flce_oracle(h, W, y, softcap=softcap, out_mult=out_mult, need_grad_h=False, need_grad_W=False)
    opred = np.asarray(ref["predicted"])
    planted = workloads.plant_labels(y, opred, 1.0 / 3.0, 7)
    counts, from_pred, _ = _all_paths(flce, h, W, planted, flags=flags, softcap=softcap, out_mult=out_mult)
    assert set(counts.values()) == {from_pred}, counts
    ref2 = flce_oracle(h, W, planted, softcap=softcap, out_mult=out_mult, need_grad_h=False, need_grad_W=False)
    valid = planted.numpy() != -100
    n_valid = int(valid.sum())
    oracle_correct = ref2["correct"]
    slack = int(np.sum((ref2["top2_gap"] < 1e-3) & valid))   # near-tie rows may go either way
    assert abs(from_pred - oracle_correct) <= slack, (from_pred, oracle_correct, slack)
    assert oracle_correct >= n_valid // 3


def test_fp32_inputs_accuracy_without_argmax(flce):
    """The fp32-input path takes the same epilogue: with and without the
    predicted tokens the counts agree."""
    N, H, V = 200, 96, 2500
    h = workloads.make_hidden(N, H, 43).float()
    W = workloads.make_weight(V, H, 43, std=0.1).float()
    y = workloads.make_labels(N, V, 43, 0.1)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    f = flce.flce_forward(hd, Wd, yd, return_predicted=True)
    torch.cuda.synchronize()
    pred = f["predicted"].cpu()
    planted = workloads.plant_labels(y, pred.numpy(), 0.5, 8).to(DEV)
    f1 = flce.flce_forward(hd, Wd, planted, return_predicted=True)
    f2 = flce.flce_forward(hd, Wd, planted, return_predicted=False)
    loss_c, acc_c = flce.flce_ce_only(hd, Wd, planted)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    c1 = _count(f1["token_accuracy"], planted.cpu())
    assert c1 == _count(f2["token_accuracy"], planted.cpu()) == _count(acc_c, planted.cpu())
    assert c1 == int(((f1["predicted"].cpu() == planted.cpu()) & (planted.cpu() != -100)).sum())
    assert c1 >= int((planted.cpu() != -100).sum()) // 2 - 1


@pytest.mark.parametrize("V", [1, 7, 300, 513])
def test_all_logits_tied(flce, V):
    """W = 0: every logit of every row is 0, so the first maximum is column 0.
    A row is correct exactly when its label is 0, on every entry point; with
    V = 1, 7 the whole vocabulary is one partial group, with 300 and 513 the
    last tile is masked."""
    N, H = 80, 64
    h = workloads.make_hidden(N, H, 44)
    W = torch.zeros((V, H), dtype=torch.bfloat16)
    y = workloads.make_labels(N, V, 44, 0.1)
    y[:7] = 0
    counts, from_pred, pred = _all_paths(flce, h, W, y)
    assert torch.all(pred == 0)
    expect = int(((y == 0) & (y != -100)).sum())
    assert from_pred == expect >= 7
    assert set(counts.values()) == {expect}, counts


def test_zero_rows_among_random_rows(flce):
    """Rows of h that are all zero have all-tied logits (first maximum 0);
    the other rows keep their own argmax; labels planted on both kinds."""
    N, H, V = 120, 96, 1100
    h = workloads.make_hidden(N, H, 45)
    W = workloads.make_weight(V, H, 45, std=0.1)
    h[::4] = 0
    y = workloads.make_labels(N, V, 45, 0.0)
    y[::8] = 0                       # zero rows labelled 0: correct
    y[4::8] = 5                      # zero rows labelled 5: wrong
    counts, from_pred, pred = _all_paths(flce, h, W, y)
    assert torch.all(pred[::4] == 0)
    assert set(counts.values()) == {from_pred}, counts
    assert from_pred >= N // 8
