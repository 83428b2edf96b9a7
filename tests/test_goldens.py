"""The stored full-size oracle results (tests/golden/configs) against the
oracle itself, on the CPU: the inputs the recipe draws here must hash to the
stored values, and a few rows recomputed by the oracle one by one must give
the stored lse, argmax and near-tie flag. This catches a stale golden file
(another recipe, another oracle) before any GPU comparison rests on it."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import oracle_rows

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "configs")
CASES = {"llama": "llama", "muse": "muse", "dsv3": "dsv3", "frozen": "frozen_ce"}


@pytest.mark.parametrize("name", sorted(CASES))
def test_golden_matches_inputs_and_oracle_rows(name):
    with open(os.path.join(GOLDEN_DIR, name + ".json")) as f:
        meta = json.load(f)
    arr = np.load(os.path.join(GOLDEN_DIR, name + ".npz"))
    w = workloads.WORKLOADS[CASES[name]]
    assert (meta["n_rows"], meta["hidden"], meta["vocab"]) == (w.n_rows, w.hidden, w.vocab)
    h, W, y = workloads.make_inputs(w)
    for k, t in (("h", h), ("W", W), ("labels", y)):
        assert workloads.tensor_sha256(t) == meta["sha256"][k], k
    n = w.n_rows
    assert all(arr[k].shape == (n,) for k in ("lse", "predicted", "top2_gap", "near_tie", "row_loss"))
    valid = y.numpy() != -100
    assert meta["n_valid"] == int(valid.sum())
    rows = np.array([0, 1, n // 2, n - 1])
    ref = oracle_rows(h[rows], W, y[rows], meta["n_valid"], softcap=w.softcap, out_mult=w.out_mult,
                      need_grad_h=False)
    # fp32-rounded stored values; the fp64 sums may differ in their last bits
    # between BLAS blockings, so allow an ulp of fp32
    np.testing.assert_allclose(arr["lse"][rows], ref["lse"], rtol=2 ** -23, atol=0)
    np.testing.assert_allclose(arr["row_loss"][rows], ref["row_loss"], rtol=2 ** -23, atol=1e-30)
    assert np.array_equal(arr["predicted"][rows], ref["predicted"].astype(np.int32))
    assert np.array_equal(arr["near_tie"][rows].astype(bool), ref["top2_gap"] < meta["near_tie_threshold"])
    # the stored batch figures are sums of the stored rows
    assert abs(float(arr["row_loss"].astype(np.float64)[valid].sum()) / meta["n_valid"] - meta["loss"]) \
        <= 1e-6 * meta["loss"]
    assert meta["near_tie_rows"] == int(arr["near_tie"].sum())
    assert meta["correct"] == int(np.sum((arr["predicted"].astype(np.int64) == y.numpy()) & valid))
