"""Pins for the CPU fp64 oracle, checked against things other than itself:
closed forms, textbook library routines (torch cross_entropy and autograd in
fp64), brute force on tiny inputs, central finite differences and invariants.
Each is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, m or T in the wrong place) fails one."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (flce_oracle, oracle_ce_logits, oracle_grad_W_rows, oracle_merge_shards, oracle_rows,
                    oracle_shard_grad_h, oracle_shard_partials)
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(n, h, v, seed, ign=1, scale=1.0):
    rng = np.random.default_rng(seed)
    hh = rng.standard_normal((n, h))
    W = rng.standard_normal((v, h)) * scale
    lab = rng.integers(0, v, n)
    lab[:ign] = -100
    return hh, W, lab


# --- 1. W = 0: every logit is 0, loss = ln V, closed-form gradients ---------------
@pytest.mark.parametrize("T", [0.0, 30.0])
@pytest.mark.parametrize("m", [1.0, 0.5])
def test_zero_weight_closed_form(T, m):
    N, H, V = 9, 6, 37
    h, _, lab = _rand(N, H, V, 1, ign=2)
    W = np.zeros((V, H))
    out = flce_oracle(h, W, lab, softcap=T, out_mult=m)
    assert out["loss"] == pytest.approx(math.log(V), rel=1e-14)
    assert np.all(out["grad_h"] == 0.0)
    # grad_W_j = m * sum_valid (1/V - [y_i = j]) h_i / n_valid
    valid = lab != -100
    nv = valid.sum()
    exp = np.zeros((V, H))
    for i in range(N):
        if not valid[i]:
            continue
        for j in range(V):
            exp[j] += m * ((1.0 / V) - (1.0 if lab[i] == j else 0.0)) * h[i] / nv
    np.testing.assert_allclose(out["grad_W"], exp, rtol=0, atol=1e-14)
    # all logits tie: argmax is the lowest index, 0
    assert np.all(out["predicted"] == 0)


def test_zero_weight_ln_v_for_the_five_heads():
    # the loss value the GPU must reproduce on W = 0 for each head's vocab
    for name, w in workloads.WORKLOADS.items():
        out = flce_oracle(np.ones((2, 8)), np.zeros((w.vocab, 8)), np.array([0, w.vocab - 1]),
                          need_grad_h=False, need_grad_W=False, block_rows=1)
        assert out["loss"] == pytest.approx(math.log(w.vocab), rel=1e-13), name


# --- 2. row sums of dlogits vanish (T = 0): read dz off grad_W with h = I ----------
def test_dlogit_row_sums_zero():
    N, V = 7, 23
    rng = np.random.default_rng(2)
    h = np.eye(N)                       # H = N, m = 1: grad_W[j, i] = dz_ij
    W = rng.standard_normal((V, N))
    lab = rng.integers(0, V, N)
    lab[3] = -100
    out = flce_oracle(h, W, lab)
    dz = out["grad_W"].T                # [N, V]
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-15)
    assert np.all(dz[3] == 0.0)
    # the label column carries (p - 1)/n_valid < 0, all others p/n_valid > 0
    for i in range(N):
        if lab[i] == -100:
            continue
        assert dz[i, lab[i]] < 0 and np.all(np.delete(dz[i], lab[i]) > 0)


def test_grad_W_column_sums_vanish_without_softcap():
    h, W, lab = _rand(11, 5, 19, 3, ign=2)
    out = flce_oracle(h, W, lab, out_mult=0.5)
    np.testing.assert_allclose(out["grad_W"].sum(axis=0), 0.0, atol=1e-14)


# --- 3. large softcap T matches no softcap ----------------------------------------
def test_large_softcap_matches_none():
    h, W, lab = _rand(12, 8, 31, 4, ign=2, scale=0.3)
    a = flce_oracle(h, W, lab, softcap=0.0)
    b = flce_oracle(h, W, lab, softcap=1e6)
    zmax = np.abs(h @ W.T).max()
    tol = 10 * (zmax / 1e6) ** 2 + 1e-13
    assert b["loss"] == pytest.approx(a["loss"], rel=tol)
    np.testing.assert_allclose(b["grad_h"], a["grad_h"], rtol=0, atol=tol * np.abs(a["grad_h"]).max())
    np.testing.assert_allclose(b["grad_W"], a["grad_W"], rtol=0, atol=tol * np.abs(a["grad_W"]).max())
    # a small cap changes the result (the cap is really applied)
    c = flce_oracle(h, W, lab, softcap=0.5)
    assert abs(c["loss"] - a["loss"]) > 1e-3


# --- 4. m identity: (m h) W^T = m (h W^T) ------------------------------------------
@pytest.mark.parametrize("T", [0.0, 2.5])
def test_out_mult_identity(T):
    h, W, lab = _rand(10, 6, 17, 5, ign=1)
    a = flce_oracle(h, W, lab, softcap=T, out_mult=0.5)
    b = flce_oracle(0.5 * h, W, lab, softcap=T, out_mult=1.0)
    assert a["loss"] == b["loss"]           # exact: 0.5 is a power of two
    np.testing.assert_array_equal(a["grad_W"], b["grad_W"])
    np.testing.assert_array_equal(a["grad_h"], 0.5 * b["grad_h"])   # chain rule through h' = m h
    # and m is really applied (not dropped)
    c = flce_oracle(h, W, lab, softcap=T, out_mult=1.0)
    assert abs(c["loss"] - a["loss"]) > 1e-6


# --- 5. central finite differences on tiny fp64 inputs ----------------------------
@pytest.mark.parametrize("T,m", [(0.0, 1.0), (2.5, 1.0), (0.0, 0.5), (2.5, 0.5)])
@pytest.mark.parametrize("red", ["mean", "sum"])
def test_finite_differences(T, m, red):
    N, H, V = 4, 5, 9
    h, W, lab = _rand(N, H, V, 6, ign=1, scale=0.7)
    g = 1.7
    out = flce_oracle(h, W, lab, softcap=T, out_mult=m, reduction=red, grad_scale=g)
    eps = 1e-6

    def L(hh, WW):
        return g * flce_oracle(hh, WW, lab, softcap=T, out_mult=m, reduction=red,
                               need_grad_h=False, need_grad_W=False)["loss"]

    fd_h = np.zeros_like(h)
    for i in range(N):
        for k in range(H):
            hp = h.copy(); hp[i, k] += eps
            hm = h.copy(); hm[i, k] -= eps
            fd_h[i, k] = (L(hp, W) - L(hm, W)) / (2 * eps)
    fd_W = np.zeros_like(W)
    for j in range(V):
        for k in range(H):
            Wp = W.copy(); Wp[j, k] += eps
            Wm = W.copy(); Wm[j, k] -= eps
            fd_W[j, k] = (L(h, Wp) - L(h, Wm)) / (2 * eps)
    np.testing.assert_allclose(out["grad_h"], fd_h, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(out["grad_W"], fd_W, rtol=1e-6, atol=1e-9)
    assert np.all(out["grad_h"][0] == 0.0)      # ignored row


# --- 6. all rows ignored ------------------------------------------------------------
def test_all_ignored():
    h, W, lab = _rand(6, 4, 11, 7, ign=6)
    G0 = np.random.default_rng(0).standard_normal((11, 4))
    out = flce_oracle(h, W, lab, softcap=3.0, grad_W0=G0)
    assert out["loss"] == 0.0 and out["token_accuracy"] == 0.0 and out["n_valid"] == 0
    assert np.all(out["grad_h"] == 0.0)
    np.testing.assert_array_equal(out["grad_W"], G0)


# --- 7. textbook routine: torch cross_entropy and autograd in fp64 ------------------
def test_matches_torch_cross_entropy_tiny_head():
    w = workloads.WORKLOADS["tiny"]
    h, W, lab = workloads.make_inputs(w)
    out = flce_oracle(h, W, lab)
    ht = h.double().requires_grad_(True)
    Wt = W.double().requires_grad_(True)
    loss = torch.nn.functional.cross_entropy(ht @ Wt.T, lab, ignore_index=-100)
    loss.backward()
    assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(out["grad_h"], ht.grad.numpy(), rtol=0,
                               atol=1e-10 * ht.grad.abs().max().item())
    np.testing.assert_allclose(out["grad_W"], Wt.grad.numpy(), rtol=0,
                               atol=1e-10 * Wt.grad.abs().max().item())


def test_softcap_gradients_match_autograd():
    N, H, V = 16, 12, 40
    h, W, lab = _rand(N, H, V, 8, ign=3, scale=0.8)
    T, m = 2.0, 0.5
    out = flce_oracle(h, W, lab, softcap=T, out_mult=m)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    # HF's capped logits: T * tanh(logits * m / T)
    logits = T * torch.tanh((ht @ Wt.T) * m / T)
    loss = torch.nn.functional.cross_entropy(logits, torch.tensor(lab), ignore_index=-100)
    loss.backward()
    assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(out["grad_h"], ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(out["grad_W"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


# --- brute force with scalar loops on a tiny case -----------------------------------
def test_brute_force_scalar_loops():
    N, H, V = 3, 2, 5
    h, W, lab = _rand(N, H, V, 9, ign=1)
    T, m = 1.5, 0.5
    tot, nv, corr = 0.0, 0, 0
    for i in range(N):
        s = []
        for j in range(V):
            z = sum(m * h[i, k] * W[j, k] for k in range(H))
            s.append(T * math.tanh(z / T))
        best = 0
        for j in range(1, V):
            if s[j] > s[best]:
                best = j
        lse = math.log(sum(math.exp(x) for x in s))
        if lab[i] != -100:
            nv += 1
            tot += lse - s[lab[i]]
            corr += int(best == lab[i])
    out = flce_oracle(h, W, lab, softcap=T, out_mult=m)
    assert out["loss"] == pytest.approx(tot / nv, rel=1e-13)
    assert out["correct"] == corr and out["token_accuracy"] == pytest.approx(corr / nv)


# --- 8. shift invariance (T = 0) -----------------------------------------------------
def test_shift_invariance():
    h, W, lab = _rand(8, 5, 13, 10, ign=1)
    a = flce_oracle(h, W, lab)
    h2 = np.concatenate([h, np.ones((8, 1))], axis=1)
    W2 = np.concatenate([W, np.full((13, 1), 3.25)], axis=1)
    b = flce_oracle(h2, W2, lab)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["grad_h"][:, :5], a["grad_h"], atol=1e-14)
    np.testing.assert_allclose(b["grad_W"][:, :5], a["grad_W"], atol=1e-14)
    np.testing.assert_array_equal(b["predicted"], a["predicted"])


# --- 9. permutation equivariance -----------------------------------------------------
def test_permutation_equivariance():
    N, H, V = 10, 6, 21
    h, W, lab = _rand(N, H, V, 11, ign=2)
    a = flce_oracle(h, W, lab, softcap=4.0)
    rng = np.random.default_rng(5)
    pv = rng.permutation(V)                 # new row j holds old row pv[j]
    inv = np.argsort(pv)
    lab2 = np.where(lab == -100, -100, inv[np.where(lab == -100, 0, lab)])
    b = flce_oracle(h, W[pv], lab2, softcap=4.0)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["grad_W"], a["grad_W"][pv], atol=1e-15)
    np.testing.assert_allclose(b["grad_h"], a["grad_h"], atol=1e-15)
    np.testing.assert_array_equal(pv[b["predicted"]], a["predicted"])
    pr = rng.permutation(N)
    c = flce_oracle(h[pr], W, lab[pr], softcap=4.0)
    assert c["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(c["grad_h"], a["grad_h"][pr], atol=1e-15)
    np.testing.assert_allclose(c["grad_W"], a["grad_W"], atol=1e-15)
    np.testing.assert_array_equal(c["lse"], a["lse"][pr])


# --- 10. closed-form grad_h (T = 0) ---------------------------------------------------
def test_closed_form_grad_h():
    N, H, V = 9, 7, 15
    h, W, lab = _rand(N, H, V, 12, ign=2)
    m = 0.5
    out = flce_oracle(h, W, lab, out_mult=m)
    p = torch.softmax(torch.tensor(m * h @ W.T), dim=1).numpy()
    nv = (lab != -100).sum()
    for i in range(N):
        if lab[i] == -100:
            np.testing.assert_array_equal(out["grad_h"][i], 0.0)
        else:
            exp = m * (p[i] @ W - W[lab[i]]) / nv
            np.testing.assert_allclose(out["grad_h"][i], exp, atol=1e-14)


# --- 11. planted accuracy --------------------------------------------------------------
def test_planted_accuracy():
    N, H, V = 64, 8, 50
    h, W, lab = _rand(N, H, V, 13, ign=6)
    pred = flce_oracle(h, W, lab, need_grad_h=False, need_grad_W=False)["predicted"]
    valid = np.nonzero(lab != -100)[0]
    rng = np.random.default_rng(1)
    plant = rng.choice(valid, size=len(valid) // 2, replace=False)
    lab2 = lab.copy()
    lab2[plant] = pred[plant]
    out = flce_oracle(h, W, lab2, need_grad_h=False, need_grad_W=False)
    natural = int(np.sum((lab2 == pred) & (lab2 != -100)))
    assert out["correct"] == natural >= len(plant)
    assert out["token_accuracy"] == pytest.approx(natural / len(valid))
    assert out["token_accuracy"] >= 0.5


def test_argmax_ties_lowest_index():
    W = np.array([[1.0, 0.0], [2.0, 0.0], [2.0, 0.0], [0.0, 1.0]])
    h = np.array([[1.0, 0.0], [0.0, 1.0]])
    out = flce_oracle(h, W, np.array([2, 3]), need_grad_h=False, need_grad_W=False)
    assert list(out["predicted"]) == [1, 3]
    assert out["correct"] == 1                      # row 0's label 2 ties with 1; lowest wins


# --- 12. += semantics of the fp32 accumulator ----------------------------------------
def test_grad_W_accumulates():
    h, W, lab = _rand(8, 4, 10, 14, ign=1)
    G0 = np.random.default_rng(3).standard_normal((10, 4))
    a = flce_oracle(h, W, lab)
    b = flce_oracle(h, W, lab, grad_W0=G0)
    np.testing.assert_allclose(b["grad_W"], G0 + a["grad_W"], atol=1e-15)


def test_sum_reduction_and_grad_scale():
    h, W, lab = _rand(8, 4, 10, 15, ign=3)
    a = flce_oracle(h, W, lab)
    b = flce_oracle(h, W, lab, reduction="sum", grad_scale=2.0)
    nv = a["n_valid"]
    assert b["loss"] == pytest.approx(a["loss"] * nv, rel=1e-14)
    np.testing.assert_allclose(b["grad_h"], a["grad_h"] * nv * 2.0, rtol=1e-13)


def test_invalid_label_rejected():
    h, W, lab = _rand(4, 3, 5, 16, ign=0)
    lab[1] = 5
    with pytest.raises(ValueError):
        flce_oracle(h, W, lab)


# --- the sampled helpers agree with the full oracle ----------------------------------
@pytest.mark.parametrize("T,m", [(0.0, 1.0), (30.0, 0.5)])
def test_sampled_helpers_agree_with_full(T, m):
    N, H, V = 40, 16, 70
    h, W, lab = _rand(N, H, V, 17, ign=4)
    full = flce_oracle(h, W, lab, softcap=T, out_mult=m)
    rows = np.array([0, 5, 17, 39])
    r = oracle_rows(h[rows], W, lab[rows], full["n_valid"], softcap=T, out_mult=m)
    np.testing.assert_allclose(r["lse"], full["lse"][rows], rtol=1e-15)
    np.testing.assert_allclose(r["grad_h"], full["grad_h"][rows], atol=1e-16)
    np.testing.assert_array_equal(r["predicted"], full["predicted"][rows])
    ids = np.array([0, 3, lab[7], 69])
    gw = oracle_grad_W_rows(h, W, lab, ids, full["lse"], full["n_valid"], softcap=T, out_mult=m,
                            block_rows=7)
    np.testing.assert_allclose(gw, full["grad_W"][ids], atol=1e-16)


@pytest.mark.parametrize("T,m", [(0.0, 1.0), (2.5, 0.5)])
def test_sampled_helpers_against_torch_autograd(T, m):
    """The sampled helpers pinned directly, not only through the full oracle:
    per-row lse, row loss and predicted token, grad_h rows and grad_W rows
    against torch's fp64 logsumexp, cross_entropy and autograd on the capped
    logits of the whole batch."""
    N, H, V = 30, 12, 45
    h, W, lab = _rand(N, H, V, 23, ign=3, scale=0.7)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = m * ht @ Wt.T
    s = T * torch.tanh(z / T) if T > 0 else z
    loss = torch.nn.functional.cross_entropy(s, torch.tensor(lab), ignore_index=-100)
    loss.backward()
    n_valid = int((lab != -100).sum())
    rows = np.array([0, 4, 11, 29])
    r = oracle_rows(h[rows], W, lab[rows], n_valid, softcap=T, out_mult=m)
    st = s.detach()
    np.testing.assert_allclose(r["lse"], torch.logsumexp(st, 1).numpy()[rows], rtol=1e-14)
    rl = torch.nn.functional.cross_entropy(st, torch.tensor(lab), ignore_index=-100, reduction="none").numpy()
    np.testing.assert_allclose(r["row_loss"], rl[rows], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(r["predicted"], st.argmax(1).numpy()[rows])
    np.testing.assert_allclose(r["grad_h"], ht.grad.numpy()[rows], rtol=1e-12, atol=1e-16)
    ids = np.array([1, 7, lab[5], 44])
    gw = oracle_grad_W_rows(h, W, lab, ids, torch.logsumexp(st, 1).numpy(), n_valid, softcap=T, out_mult=m,
                            block_rows=8)
    np.testing.assert_allclose(gw, Wt.grad.numpy()[ids], rtol=1e-12, atol=1e-16)


# --- the pages' printed accumulator sizes pin fp32 [V, H] ----------------------------
def test_page_accumulator_sizes():
    with open(os.path.join(GOLDEN, "page_figures.json")) as f:
        figs = json.load(f)["fp32_grad_weight_accumulator"]
    for fg in figs:
        nbytes = fg["vocab"] * fg["hidden"] * 4
        assert round(nbytes / fg["unit_bytes"], fg["decimals"]) == fg["value_printed"]
        if "bf16_value_printed" in fg:
            assert round(nbytes / 2 / fg["unit_bytes"], fg["decimals"]) == fg["bf16_value_printed"]


def test_workload_recipe_is_deterministic_and_shaped():
    w = workloads.WORKLOADS["tiny"]
    h1, W1, l1 = workloads.make_inputs(w)
    h2, W2, l2 = workloads.make_inputs(w)
    assert torch.equal(h1, h2) and torch.equal(W1, W2) and torch.equal(l1, l2)
    assert h1.dtype == torch.bfloat16 and W1.shape == (4096, 512)
    assert int((l1 == -100).sum()) == round(0.10 * 256)
    assert abs(W1.float().std().item() - 0.02) < 1e-3
    z = workloads.make_labels(20000, 1000, 3, 0.03, "zipf", 1.1)
    zv = z[z != -100]
    assert int((z == -100).sum()) == 600
    # Zipf(1.1): id 0 is the most frequent, about 1/H_{1000,1.1} of the draws
    hz = sum((k + 1) ** -1.1 for k in range(1000))
    assert abs(float((zv == 0).float().mean()) - 1 / hz) < 0.02


def test_input_generator_is_splitmix64():
    """The input streams are SplitMix64: its published first outputs for seed
    1234567 (the test vector of the reference C implementation)."""
    got = workloads.draws(np.uint64(1234567), 0, 5)
    assert [int(x) for x in got] == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                     4593380528125082431, 16408922859458223821]
    # draws are addressed by index: a window equals the same slice of a longer run
    key = np.uint64(99)
    assert np.array_equal(workloads.draws(key, 1000, 7), workloads.draws(key, 0, 1007)[1000:])
    # normals: mean 0, variance 1, and a block boundary does not change them
    h = workloads.make_hidden(2048, 4096, 5).float()
    assert abs(h.mean().item()) < 5e-3 and abs(h.std().item() - 1.0) < 5e-3
    assert torch.equal(workloads.make_hidden(3, 4096, 5), workloads.make_hidden(2048, 4096, 5)[:3])


# --- cross-entropy on materialised logits -------------------------------------------
def test_ce_logits_matches_torch_and_autograd():
    from oracle import oracle_ce_logits
    rng = np.random.default_rng(20)
    N, V = 37, 53
    x = rng.standard_normal((N, V)) * 3
    lab = rng.integers(0, V, N)
    lab[[2, 9]] = -100
    for T, m in [(0.0, 1.0), (2.5, 0.5)]:
        xt = torch.tensor(x, requires_grad=True)
        s = T * torch.tanh(xt * m / T) if T > 0 else xt * m
        loss = torch.nn.functional.cross_entropy(s, torch.tensor(lab), ignore_index=-100)
        loss.backward()
        out = oracle_ce_logits(x, lab, softcap=T, out_mult=m)
        assert out["loss"] == pytest.approx(loss.item(), rel=1e-13)
        np.testing.assert_allclose(out["grad_logits"], xt.grad.numpy(), rtol=1e-12, atol=1e-15)
        # reduction none: per-row losses of torch, and the gradient of sum_i r_i l_i
        xt2 = torch.tensor(x, requires_grad=True)
        s2 = T * torch.tanh(xt2 * m / T) if T > 0 else xt2 * m
        rl = torch.nn.functional.cross_entropy(s2, torch.tensor(lab), ignore_index=-100, reduction="none")
        r = torch.tensor(rng.standard_normal(N))
        (rl * r).sum().backward()
        o2 = oracle_ce_logits(x, lab, softcap=T, out_mult=m, reduction="none", row_scale=r.numpy())
        np.testing.assert_allclose(o2["row_loss"], rl.detach().numpy(), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o2["grad_logits"], xt2.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_ce_logits_equals_fused_with_identity_weight():
    from oracle import oracle_ce_logits
    rng = np.random.default_rng(21)
    N, V = 24, 31
    x = rng.standard_normal((N, V))
    lab = rng.integers(0, V, N)
    lab[0] = -100
    a = oracle_ce_logits(x, lab, softcap=4.0, out_mult=0.5)
    b = flce_oracle(x, np.eye(V), lab, softcap=4.0, out_mult=0.5)   # h = logits, W = I
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["grad_logits"], b["grad_h"], atol=1e-16)
    np.testing.assert_array_equal(a["predicted"], b["predicted"])


# --- randomised: finite differences and the textbook routine on drawn shapes -------
def test_randomised_gradients_and_loss_against_autograd():
    """Hypothesis draws small shapes, softcaps, multipliers (negative too),
    reductions and ignored rows; the oracle's loss must equal torch's
    cross_entropy on the fp64 capped logits, and its gradients fp64 autograd
    through the same expression (an implementation that shares nothing with
    the oracle's closed-form backward)."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    import torch

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(N=st.integers(1, 6), H=st.integers(1, 7), V=st.integers(2, 12),
               T=st.sampled_from([0.0, 0.3, 2.5, 30.0]), m=st.sampled_from([1.0, 0.5, -1.25, 3.0]),
               red=st.sampled_from(["mean", "sum"]), seed=st.integers(0, 10_000))
    def check(N, H, V, T, m, red, seed):
        rng = np.random.default_rng(seed)
        h = rng.standard_normal((N, H))
        W = rng.standard_normal((V, H)) * 0.8
        lab = rng.integers(0, V, N)
        lab[rng.random(N) < 0.25] = -100
        out = flce_oracle(h, W, lab, softcap=T, out_mult=m, reduction=red, grad_scale=1.3)
        ht = torch.tensor(h, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        z = m * (ht @ Wt.T)
        s = T * torch.tanh(z / T) if T > 0 else z
        y = torch.tensor(lab)
        if (y != -100).any():
            loss = torch.nn.functional.cross_entropy(s, y, ignore_index=-100, reduction=red)
            (1.3 * loss).backward()
            assert abs(out["loss"] - loss.item()) <= 1e-12 * max(1.0, abs(loss.item()))
            np.testing.assert_allclose(out["grad_h"], ht.grad.numpy(), rtol=1e-10, atol=1e-13)
            np.testing.assert_allclose(out["grad_W"], Wt.grad.numpy(), rtol=1e-10, atol=1e-13)
        else:
            assert out["loss"] == 0.0 and not out["grad_h"].any() and not out["grad_W"].any()
        pred = s.detach().numpy().argmax(1)             # numpy's argmax takes the first maximum
        np.testing.assert_array_equal(out["predicted"], pred)

    check()


# --- top-2 gap: the rule that excuses near-tie rows from the predicted-token check ---
# The gap of row i is (s1 - s2) / |s1|, s1 >= s2 the two largest capped logits
# counted with multiplicity (a repeated maximum gives gap 0). These pins fix the
# second-largest index (not the smallest or the maximum again), the absolute
# value in the denominator, duplicates, and that the gap is taken on s = cap(m z),
# not on z.
def _gap_brute(s_row):
    srt = sorted(s_row, reverse=True)
    return (srt[0] - srt[1]) / abs(srt[0])


def _logit_rows(c_rows):
    """h = e_0 and W[j] = c_j e_0, so z_ij = c_ij exactly (one row per case)."""
    c = np.asarray(c_rows, dtype=np.float64)
    V = c.shape[1]
    out = []
    for row in c:
        W = np.zeros((V, 3))
        W[:, 0] = row
        out.append((np.array([[1.0, 0.0, 0.0]]), W))
    return out


@pytest.mark.parametrize("case,expect", [
    ([1.0, 5.0, 3.0, -2.0], 0.4),        # clear winner: (5 - 3) / 5
    ([-3.0, -1.0, -2.0], 1.0),           # negative maximum: (-1 - -2) / |-1|
    ([5.0, 5.0, 3.0], 0.0),              # repeated maximum counts twice
    ([2.0, 7.0, 7.0, 7.0], 0.0),
    ([0.25, -0.5, 0.125, 0.0], 0.5),     # (0.25 - 0.125) / 0.25
])
def test_top2_gap_closed_forms(case, expect):
    (h, W), = _logit_rows([case])
    for out in (flce_oracle(h, W, np.array([0]), need_grad_h=False, need_grad_W=False),
                oracle_rows(h, W, np.array([0]), 1, need_grad_h=False),
                oracle_ce_logits(np.array([case]), np.array([0]), need_grad=False)):
        assert out["top2_gap"][0] == pytest.approx(expect, abs=1e-15)
        assert out["predicted"][0] == int(np.argmax(case))


def test_top2_gap_is_taken_on_capped_and_scaled_logits():
    (h, W), = _logit_rows([[10.0, 20.0, -4.0]])
    T, m = 5.0, 0.5
    s = [T * math.tanh(m * c / T) for c in (10.0, 20.0, -4.0)]
    out = flce_oracle(h, W, np.array([1]), softcap=T, out_mult=m, need_grad_h=False, need_grad_W=False)
    assert out["top2_gap"][0] == pytest.approx(_gap_brute(s), rel=1e-14)
    # on the raw z the gap would be (20 - 10) / 20 = 0.5, on m z also 0.5
    assert abs(out["top2_gap"][0] - 0.5) > 0.1


def test_top2_gap_exact_tie_between_identical_vocab_rows():
    rng = np.random.default_rng(21)
    N, H, V = 6, 5, 17
    h = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H))
    out0 = flce_oracle(h, W, np.zeros(N, dtype=np.int64), need_grad_h=False, need_grad_W=False)
    # copy each row's winning vocab row to a higher index: an exact tie, gap 0,
    # and the lowest index must still win
    W2 = np.concatenate([W, W[out0["predicted"][:1]]], axis=0)
    out = flce_oracle(h, W2, np.zeros(N, dtype=np.int64), need_grad_h=False, need_grad_W=False)
    assert out["top2_gap"][0] == 0.0
    assert out["predicted"][0] == out0["predicted"][0]


@pytest.mark.parametrize("T,m", [(0.0, 1.0), (3.0, 0.5), (0.0, -1.5)])
def test_top2_gap_brute_force_sorted_rows(T, m):
    rng = np.random.default_rng(22)
    N, H, V = 11, 4, 9
    h = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H))
    out = flce_oracle(h, W, np.zeros(N, dtype=np.int64), softcap=T, out_mult=m,
                      need_grad_h=False, need_grad_W=False)
    for i in range(N):
        s = []
        for j in range(V):
            z = sum(m * h[i, k] * W[j, k] for k in range(H))
            s.append(T * math.tanh(z / T) if T > 0 else z)
        assert out["top2_gap"][i] == pytest.approx(_gap_brute(s), rel=1e-12, abs=1e-15)


def test_top2_gap_single_column_vocab_is_infinite():
    out = flce_oracle(np.ones((2, 3)), np.ones((1, 3)), np.array([0, -100]), need_grad_h=False, need_grad_W=False)
    assert np.all(np.isinf(out["top2_gap"]))


# --- vocabulary shards: per-shard partials, their merge, per-shard grad_h ------------
def _torch_capped(h, W, T, m):
    z = m * (torch.tensor(h) @ torch.tensor(W).T)
    return T * torch.tanh(z / T) if T > 0 else z


@pytest.mark.parametrize("offsets", [[0, 23], [0, 5, 13, 23], [0, 1, 2, 22, 23]])
@pytest.mark.parametrize("T,m", [(0.0, 1.0), (4.0, 0.5)])
def test_shard_partials_against_torch_slices(offsets, T, m):
    N, H, V = 9, 6, 23
    h, W, lab = _rand(N, H, V, 40, ign=2)
    part = oracle_shard_partials(h, W, lab, offsets, softcap=T, out_mult=m)
    s = _torch_capped(h, W, T, m)
    for k in range(len(offsets) - 1):
        sk = s[:, offsets[k]:offsets[k + 1]]
        np.testing.assert_allclose(part["max"][k], sk.max(dim=1).values.numpy(), rtol=0, atol=1e-14)
        lse_k = torch.logsumexp(sk, dim=1).numpy()
        np.testing.assert_allclose(part["max"][k] + np.log(part["sumexp"][k]), lse_k, rtol=1e-14)
        np.testing.assert_array_equal(part["argmax"][k], offsets[k] + sk.argmax(dim=1).numpy())
        for i in range(N):
            inside = lab[i] != -100 and offsets[k] <= lab[i] < offsets[k + 1]
            assert part["target"][k][i] == pytest.approx(float(s[i, lab[i]]) if inside else 0.0, rel=1e-14, abs=0)


@pytest.mark.parametrize("offsets", [[0, 23], [0, 5, 13, 23], [0, 11, 12, 23]])
@pytest.mark.parametrize("T,m", [(0.0, 1.0), (4.0, 0.5)])
def test_merged_shards_match_torch_on_the_full_vocabulary(offsets, T, m):
    N, H, V = 12, 5, 23
    h, W, lab = _rand(N, H, V, 41, ign=3)
    part = oracle_shard_partials(h, W, lab, offsets, softcap=T, out_mult=m)
    out = oracle_merge_shards(part, lab, offsets)
    s = _torch_capped(h, W, T, m)
    np.testing.assert_allclose(out["lse"], torch.logsumexp(s, dim=1).numpy(), rtol=1e-14)
    np.testing.assert_array_equal(out["predicted"], s.argmax(dim=1).numpy())
    ref = torch.nn.functional.cross_entropy(s, torch.tensor(lab), ignore_index=-100)
    assert out["loss"] == pytest.approx(ref.item(), rel=1e-13)
    assert out["n_valid"] == int((lab != -100).sum())


def test_merged_shards_tie_across_shards_keeps_lowest_id():
    # vocab row 3 (shard 0) copied to vocab row 17 (shard 2): an exact tie
    # across shards for every row whose winner is row 3
    N, H, V = 16, 4, 20
    rng = np.random.default_rng(42)
    h = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H))
    W[3] = 3.0 * np.abs(W[3]).max() * np.sign(h.mean(axis=0))
    W[17] = W[3]
    lab = np.full(N, 17)
    offsets = [0, 8, 12, 20]
    out = oracle_merge_shards(oracle_shard_partials(h, W, lab, offsets), lab, offsets)
    full = flce_oracle(h, W, lab, need_grad_h=False, need_grad_W=False)
    assert np.sum(full["predicted"] == 3) >= 4
    np.testing.assert_array_equal(out["predicted"], full["predicted"])
    assert out["correct"] == 0


@pytest.mark.parametrize("T,m", [(0.0, 1.0), (3.0, 0.5)])
def test_shard_grad_h_parts_sum_to_autograd(T, m):
    N, H, V = 7, 5, 19
    h, W, lab = _rand(N, H, V, 43, ign=2)
    ht = torch.tensor(h, requires_grad=True)
    z = m * (ht @ torch.tensor(W).T)
    s = T * torch.tanh(z / T) if T > 0 else z
    torch.nn.functional.cross_entropy(s, torch.tensor(lab), ignore_index=-100).backward()
    lse = torch.logsumexp(s.detach(), dim=1).numpy()
    nv = int((lab != -100).sum())
    offsets = [0, 4, 11, 19]
    parts = [oracle_shard_grad_h(h, W, lab, lse, nv, offsets[k], offsets[k + 1], softcap=T, out_mult=m)
             for k in range(3)]
    np.testing.assert_allclose(sum(parts), ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    # a shard holding none of the labels contributes m sum_j p_ij W_j (T = 0) alone
    if T == 0.0:
        p = torch.softmax(s.detach(), dim=1).numpy()
        k = 1
        sel = (lab == -100) | (lab < offsets[k]) | (lab >= offsets[k + 1])
        exp = m * (p[:, offsets[k]:offsets[k + 1]] @ W[offsets[k]:offsets[k + 1]]) / nv
        exp[lab == -100] = 0.0
        np.testing.assert_allclose(parts[k][sel], exp[sel], atol=1e-14)
