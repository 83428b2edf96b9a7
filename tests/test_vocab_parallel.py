"""Vocabulary-parallel FLCE on one GPU: W split by vocabulary rows into S
shards, each run as its own pair of calls (flce_vp_forward, then
flce_vp_backward on the gathered partials), one after another on one GPU. The
partials of each shard are compared with the oracle's shard partials; the
merged outputs with the unsharded call (predictions bit for bit: the argmax
merge is exact) and with the fp64 oracle at the library's tolerances; grad_h
summed over the shards and every shard's grad_W with the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle, oracle_rows, oracle_shard_partials

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _inputs(N, H, V, seed, ign=0.1, std=0.05):
    return (workloads.make_hidden(N, H, seed), workloads.make_weight(V, H, seed, std=std),
            workloads.make_labels(N, V, seed, ign))


def _run_shards(flce, h, W, y, offsets, grad_h=True, grad_W=True, stored=False, **kw):
    """Every shard's forward, the gather (stacking in shard order), every
    shard's backward; returns the partials, the first shard's outputs, the
    summed grad_h (bf16, rounded by the library) and the full grad_W. With
    stored, each shard keeps its logits between its two calls
    (FLCE_FLAG_VP_STORED) in a workspace of its own."""
    V = offsets[-1]
    hd, yd = h.to(DEV), y.to(DEV)
    if stored:
        kw = dict(kw, flags=kw.get("flags", 0) | flce.FLCE_FLAG_VP_STORED)
    fwd_kw = {k: v for k, v in kw.items() if k in ("softcap", "out_mult", "chunk_rows", "flags")}
    shards = [W[offsets[k]:offsets[k + 1]].to(DEV) for k in range(len(offsets) - 1)]
    wss = [flce.flce_vp_workspace(hd, Wk, keep_logits=True) if stored else None for Wk in shards]
    parts = [flce.flce_vp_forward(hd, Wk, yd, offsets[k], V, workspace=wss[k], **fwd_kw)
             for k, Wk in enumerate(shards)]
    allp = torch.stack(parts)
    gh32 = torch.zeros((h.shape[0], h.shape[1]), dtype=torch.float32, device=DEV) if grad_h else None
    gW = torch.zeros((V, h.shape[1]), dtype=torch.float32, device=DEV) if grad_W else None
    outs = []
    for k, Wk in enumerate(shards):
        outs.append(flce.flce_vp_backward(hd, Wk, yd, allp, offsets, offsets[k], V, grad_h_partial=gh32,
                                          grad_W=None if gW is None else gW[offsets[k]:offsets[k + 1]],
                                          return_lse=True, workspace=wss[k], **kw))
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    for ws in wss:
        assert ws is None or flce.flce_get_status(workspace=ws) == 0
    gh = flce.flce_scale_gradient(gh32, None, out_dtype=torch.bfloat16) if grad_h else None
    return allp, outs, gh, gW


CASES = [
    dict(N=300, H=128, V=3001, offsets=[0, 3001], seed=51),
    dict(N=300, H=128, V=3001, offsets=[0, 1700, 3001], seed=52),
    dict(N=700, H=192, V=5000, offsets=[0, 1024, 3333, 5000], seed=53, softcap=30.0, out_mult=0.5),
    dict(N=1030, H=256, V=4099, offsets=[0, 7, 4000, 4099], seed=54, chunk_rows=256),
]


@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "stored"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{len(c['offsets']) - 1}-N{c['N']}-V{c['V']}")
def test_shards_match_oracle_and_unsharded(flce, case, stored):
    N, H, V, offsets = case["N"], case["H"], case["V"], case["offsets"]
    kw = {k: case[k] for k in ("softcap", "out_mult", "chunk_rows") if k in case}
    okw = {k: case[k] for k in ("softcap", "out_mult") if k in case}
    h, W, y = _inputs(N, H, V, case["seed"])
    allp, outs, gh, gW = _run_shards(flce, h, W, y, offsets, stored=stored, **kw)

    # each shard's partials against the oracle's
    ref_p = oracle_shard_partials(h, W, y, offsets, **okw)
    got = allp.cpu()
    S = len(offsets) - 1
    mx = got[:, 0].double().numpy()
    assert np.abs(mx - ref_p["max"]).max() <= 1e-4 * np.abs(ref_p["max"]).max()
    lse_k = mx + np.log(got[:, 1].double().numpy())
    ref_lse_k = ref_p["max"] + np.log(ref_p["sumexp"])
    assert np.abs(lse_k - ref_lse_k).max() <= 1e-4 * np.abs(ref_lse_k).max()
    arg = got[:, 2].contiguous().view(torch.int32).numpy()
    # argmax within a shard: exact unless the shard's own top two nearly tie
    for k in range(S):
        assert np.all((arg[k] >= offsets[k]) & (arg[k] < offsets[k + 1]))
    tgt = got[:, 3].double().numpy()
    assert np.abs(tgt - ref_p["target"]).max() <= 1e-4 * max(1.0, np.abs(ref_p["target"]).max())

    # merged outputs: the same on every shard
    for o in outs[1:]:
        assert float(o["loss"]) == float(outs[0]["loss"]) and torch.equal(o["predicted"], outs[0]["predicted"])
        assert torch.equal(o["lse"], outs[0]["lse"])
    # against the unsharded call: predictions bit for bit, lse to fp32 merge order
    f = flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV), return_lse=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(outs[0]["predicted"], f["predicted"])
    assert float(outs[0]["token_accuracy"]) == float(f["token_accuracy"])
    assert (outs[0]["lse"] - f["lse"]).abs().max().item() <= 1e-5 * f["lse"].abs().max().item()
    # against the oracle
    ref = flce_oracle(h, W, y, **okw)
    assert abs(float(outs[0]["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    near = ref["top2_gap"] < 1e-3
    pred = outs[0]["predicted"].cpu().numpy()
    assert np.all((pred == ref["predicted"]) | near)
    g = gh.float().cpu().numpy()
    assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * np.abs(ref["grad_h"]).max()
    gw = gW.double().cpu().numpy()
    assert np.abs(gw - ref["grad_W"]).max() <= 1e-2 * np.abs(ref["grad_W"]).max()


@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "stored"])
def test_two_shards_of_the_dsv3_head(flce, stored):
    """The DeepSeek-V3-shaped head (H = 7168, V = 129280) on 4096 rows in two
    vocab shards: merged loss and predictions against the unsharded low-memory
    call, grad_h and grad_W against it at bf16 rounding, and sampled rows against
    the oracle."""
    w = workloads.WORKLOADS["dsv3"]
    N = 4096
    h, W, y = workloads.make_inputs(w, n_rows=N)
    offsets = [0, 64640, w.vocab]
    allp, outs, gh, gW = _run_shards(flce, h, W, y, offsets, stored=stored)
    gW1 = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
    o = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW1, return_predicted=True,
                                   low_memory=True)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    assert torch.equal(outs[0]["predicted"], o["predicted"])
    assert abs(float(outs[0]["loss"]) - float(o["loss"])) <= 1e-6 * abs(float(o["loss"]))
    assert float(outs[0]["token_accuracy"]) == float(o["token_accuracy"])
    x, z = gh.float(), o["grad_h"].float()
    assert (x - z).abs().max().item() <= 2.0 ** -7 * z.abs().max().item()
    assert (gW - gW1).abs().max().item() <= 1e-3 * gW1.abs().max().item()
    n_valid = int((y != -100).sum())
    rows = workloads.sample_indices(N, 64, seed=400)
    ref = oracle_rows(h[rows], W, y[rows], n_valid)
    g = gh[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * np.abs(ref["grad_h"]).max()
    flce.flce_release_workspaces()


@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "stored"])
def test_forward_only_and_frozen_shards(flce, stored):
    """A backward with neither gradient (loss and predictions only) and one
    with grad_W alone (grad_h not wanted)."""
    N, H, V = 500, 64, 2500
    h, W, y = _inputs(N, H, V, 55)
    offsets = [0, 1200, 2500]
    _, outs, gh, gW = _run_shards(flce, h, W, y, offsets, grad_h=False, grad_W=False, stored=stored)
    assert gh is None and gW is None
    ref = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=False)
    assert abs(float(outs[0]["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    _, outs2, gh2, gW2 = _run_shards(flce, h, W, y, offsets, grad_h=False, grad_W=True, stored=stored)
    assert float(outs2[0]["loss"]) == float(outs[0]["loss"])
    ref = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=True)
    gw = gW2.double().cpu().numpy()
    assert np.abs(gw - ref["grad_W"]).max() <= 1e-2 * np.abs(ref["grad_W"]).max()


def test_bad_labels_and_shard_tables(flce):
    from linear_cross_entropy_02_gb300 import _lib
    N, H, V = 64, 32, 600
    h, W, y = _inputs(N, H, V, 56)
    y[5] = V + 3                              # outside [0, vocab_total)
    hd, yd = h.to(DEV), y.to(DEV)
    parts = [flce.flce_vp_forward(hd, W[a:b].to(DEV), yd, a, V) for a, b in ((0, 300), (300, 600))]
    torch.cuda.synchronize()
    assert flce.flce_get_status() & _lib.FLCE_ERR_LABEL
    allp = torch.stack(parts)
    for bad in ([0, 300], [0, 300, 601], [1, 300, 600], [0, 400, 600], [0, 300, 300, 600]):
        with pytest.raises(flce.FlceError) as e:
            flce.flce_vp_backward(hd, W[0:300].to(DEV), yd, allp[:len(bad) - 1] if len(bad) == 3 else
                                  allp[:1].expand(len(bad) - 1, 4, N).contiguous(), bad, 0, V)
        assert e.value.code == _lib.FLCE_ERR_ARG
    flce.flce_release_workspaces()


def _fuzz(n=10, seed=90):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        V = int(rng.integers(300, 6000))
        S = int(rng.integers(1, 5))
        cuts = sorted(set(int(x) for x in rng.integers(1, V, S - 1))) if S > 1 else []
        out.append(dict(N=int(rng.integers(1, 900)), H=int(8 * rng.integers(1, 40)), V=V, offsets=[0] + cuts + [V],
                        softcap=float(rng.choice([0.0, 2.0, 30.0])), out_mult=float(rng.choice([1.0, 0.5, -1.5])),
                        chunk_rows=int(rng.choice([0, 128, 384])), vocab_slab=int(rng.choice([0, 256, 1024])),
                        seed=100 + i))
    return out


@pytest.mark.parametrize("case", _fuzz(), ids=lambda c: f"N{c['N']}-H{c['H']}-V{c['V']}-S{len(c['offsets']) - 1}")
@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "stored"])
def test_fuzzed_shard_tables(flce, case, stored):
    """Seeded random shapes, options and shard boundaries (none aligned to the
    256-column tiles), against the fp64 oracle and the unsharded call, in both
    backward forms."""
    kw = {k: case[k] for k in ("softcap", "out_mult", "chunk_rows")}
    okw = {k: case[k] for k in ("softcap", "out_mult")}
    h, W, y = _inputs(case["N"], case["H"], case["V"], case["seed"])
    _, outs, gh, gW = _run_shards(flce, h, W, y, case["offsets"], vocab_slab=case["vocab_slab"], stored=stored,
                                  **kw)
    f = flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV), **kw)
    torch.cuda.synchronize()
    assert torch.equal(outs[0]["predicted"], f["predicted"])
    assert float(outs[0]["token_accuracy"]) == float(f["token_accuracy"])
    ref = flce_oracle(h, W, y, **okw)
    if ref["n_valid"]:
        assert abs(float(outs[0]["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    g = gh.float().cpu().numpy()
    assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * max(np.abs(ref["grad_h"]).max(), 1e-30)
    gw = gW.double().cpu().numpy()
    assert np.abs(gw - ref["grad_W"]).max() <= 1e-2 * max(np.abs(ref["grad_W"]).max(), 1e-30)


@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "stored"])
def test_empty_and_all_ignored_batches(flce, stored):
    """No rows, and rows that are all ignored: the loss and accuracy are 0, the
    gradients stay 0 and nothing reads outside the (empty) inputs."""
    H, V = 64, 1000
    offsets = [0, 400, V]
    W = workloads.make_weight(V, H, 57)
    for N, ign in ((0, 0.0), (70, 1.0)):
        h = workloads.make_hidden(max(N, 1), H, 57)[:N]
        y = workloads.make_labels(max(N, 1), V, 57, ign)[:N]
        _, outs, gh, gW = _run_shards(flce, h, W, y, offsets, stored=stored)
        assert float(outs[0]["loss"]) == 0.0 and float(outs[0]["token_accuracy"]) == 0.0
        assert torch.count_nonzero(gh).item() == 0 and torch.count_nonzero(gW).item() == 0


def test_stored_and_recomputed_shards_agree(flce):
    """The two backward forms of the same shards: the forward outputs (the
    partials, then the merged loss, accuracy, predictions and lse) are the
    same bits, since the forward GEMM's statistics do not depend on whether
    the logits are also stored; the gradients agree to the bf16 rounding of
    dz, taken from fp16 stored logits in one form and fp32 recomputed ones in
    the other."""
    N, H, V = 900, 192, 6000
    h, W, y = _inputs(N, H, V, 57)
    offsets = [0, 2048, 4000, 6000]
    kw = dict(softcap=30.0, out_mult=0.5)
    p1, o1, gh1, gW1 = _run_shards(flce, h, W, y, offsets, **kw)
    p2, o2, gh2, gW2 = _run_shards(flce, h, W, y, offsets, stored=True, **kw)
    assert torch.equal(p1, p2)
    for a, b in zip(o1, o2):
        assert float(a["loss"]) == float(b["loss"]) and float(a["token_accuracy"]) == float(b["token_accuracy"])
        assert torch.equal(a["predicted"], b["predicted"]) and torch.equal(a["lse"], b["lse"])
    assert (gh1.float() - gh2.float()).abs().max().item() <= 2.0 ** -6 * gh1.float().abs().max().item()
    assert (gW1 - gW2).abs().max().item() <= 1e-2 * gW1.abs().max().item()


def test_stored_shard_needs_its_workspace(flce):
    """FLCE_FLAG_VP_STORED without an explicit workspace is refused on the
    host: the cached one could be reused between the two calls."""
    N, H, V = 64, 32, 600
    h, W, y = _inputs(N, H, V, 58)
    with pytest.raises(ValueError):
        flce.flce_vp_forward(h.to(DEV), W[:300].to(DEV), y.to(DEV), 0, V, flags=flce.FLCE_FLAG_VP_STORED)
