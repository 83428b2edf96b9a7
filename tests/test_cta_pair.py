"""GEMMs on CTA pairs (FLCE_FLAG_CTA_PAIR): each 256 x 256 tile is computed by
a cluster of two CTAs with tcgen05 cta_group::2, every CTA holding 128 rows in
a double-buffered TMEM accumulator. Checked against the fp64 oracle at the
library's tolerances, and against the single-CTA 256 x 256 tiles, which add the
same products in the same K order."""
import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle
from test_parity import check_against_oracle, run_fwd_bwd

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
PAIR = 64
TILE256 = 32
RECOMPUTE = 8


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def _inputs(N, H, V, seed, ign=0.1, std=0.05):
    return (workloads.make_hidden(N, H, seed), workloads.make_weight(V, H, seed, std=std),
            workloads.make_labels(N, V, seed, ign))


def _same(a, b, what):
    assert float(a["loss"]) == float(b["loss"]), what
    assert torch.equal(a["predicted"], b["predicted"]), what
    assert torch.equal(a["grad_h"], b["grad_h"]), what
    if a["grad_W"] is not None:
        assert torch.equal(a["grad_W"], b["grad_W"]), what


def test_pair_tiny_head(flce):
    w = workloads.WORKLOADS["tiny"]
    h, W, y = workloads.make_inputs(w)
    out = run_fwd_bwd(flce, h, W, y, flags=TILE256 | PAIR)
    ref = flce_oracle(h, W, y)
    check_against_oracle(out, ref, y, what="tiny pair")
    _same(out, run_fwd_bwd(flce, h, W, y, flags=TILE256), "tiny pair vs single-CTA 256-row tiles")


@pytest.mark.parametrize("extra", [0, RECOMPUTE])
@pytest.mark.parametrize("case", [
    dict(N=300, H=192, V=1000, chunk_rows=128),      # one 128-row tile: the follower's rows lie past M
    dict(N=513, H=136, V=777, chunk_rows=256, softcap=30.0, out_mult=0.5),
    dict(N=1100, H=192, V=1500, chunk_rows=768),
    dict(N=2048, H=512, V=5003, softcap=2.0, out_mult=0.5, reduction="sum", grad_scale=0.75),
])
def test_pair_edge_shapes(flce, case, extra):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h, W, y = _inputs(N, H, V, 71)
    out = run_fwd_bwd(flce, h, W, y, flags=TILE256 | PAIR | extra, **c)
    ref = flce_oracle(h, W, y, **{k: v for k, v in c.items() if k != "chunk_rows"})
    check_against_oracle(out, ref, y, what=f"pair {case} {extra}")
    _same(out, run_fwd_bwd(flce, h, W, y, flags=TILE256 | extra, **c), f"pair vs single {case} {extra}")


def test_pair_full_dsv3_head(flce):
    """The DeepSeek-V3 head in the benchmark's configuration: pairs against
    single-CTA 256-row tiles, every output."""
    w = workloads.WORKLOADS["dsv3"]
    h, W, y = workloads.make_inputs(w)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    outs = []
    for flags in (0, PAIR):
        gW = torch.zeros(W.shape, dtype=torch.float32, device=DEV)
        o = flce.flce_forward_backward(hd, Wd, yd, grad_W=gW, return_predicted=True, flags=flags)
        torch.cuda.synchronize()
        assert flce.flce_get_status() == 0
        outs.append(o)
        flce.flce_release_workspaces()
    _same(outs[0], outs[1], "dsv3 pair vs single")


def test_pair_ce_only_and_vocab_shards(flce):
    N, H, V = 1500, 256, 9000
    h, W, y = _inputs(N, H, V, 72)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    a = flce.flce_ce_only(hd, Wd, yd, flags=TILE256 | PAIR)
    b = flce.flce_ce_only(hd, Wd, yd, flags=TILE256)
    torch.cuda.synchronize()
    assert float(a[0]) == float(b[0]) and float(a[1]) == float(b[1])
    offsets = [0, 4000, V]
    parts = [flce.flce_vp_forward(hd, Wd[offsets[k]:offsets[k + 1]], yd, offsets[k], V, flags=TILE256 | PAIR)
             for k in range(2)]
    allp = torch.stack(parts)
    gh = torch.zeros((N, H), dtype=torch.float32, device=DEV)
    for k in range(2):
        o = flce.flce_vp_backward(hd, Wd[offsets[k]:offsets[k + 1]], yd, allp, offsets, offsets[k], V,
                                  grad_h_partial=gh, flags=TILE256 | PAIR)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, need_grad_W=False)
    assert abs(float(o["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    g = gh.double().cpu().numpy()
    assert np.abs(g - ref["grad_h"]).max() <= 1e-2 * np.abs(ref["grad_h"]).max()


def test_pair_vocab_shards_with_kept_logits(flce):
    """Vocab shards that keep their logits between their calls
    (FLCE_FLAG_VP_STORED), on CTA pairs and on single CTAs: the same bits
    (the same products in the same K order), and the oracle's values."""
    from linear_cross_entropy_02_gb300 import _lib
    N, H, V = 1500, 256, 9000
    h, W, y = _inputs(N, H, V, 73)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    offsets = [0, 4000, V]
    res = []
    for flags in (TILE256 | PAIR | _lib.FLCE_FLAG_VP_STORED, TILE256 | _lib.FLCE_FLAG_VP_STORED):
        shards = [Wd[offsets[k]:offsets[k + 1]] for k in range(2)]
        wss = [flce.flce_vp_workspace(hd, shards[k], keep_logits=True, chunk_rows=512) for k in range(2)]
        parts = [flce.flce_vp_forward(hd, shards[k], yd, offsets[k], V, flags=flags, chunk_rows=512,
                                      workspace=wss[k]) for k in range(2)]
        allp = torch.stack(parts)
        gh = torch.zeros((N, H), dtype=torch.float32, device=DEV)
        gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
        for k in range(2):
            o = flce.flce_vp_backward(hd, shards[k], yd, allp, offsets, offsets[k], V, grad_h_partial=gh,
                                      grad_W=gW[offsets[k]:offsets[k + 1]], flags=flags, chunk_rows=512,
                                      workspace=wss[k])
        torch.cuda.synchronize()
        assert all(flce.flce_get_status(workspace=ws) == 0 for ws in wss)
        res.append((allp, o, gh, gW))
    (p1, o1, gh1, gW1), (p2, o2, gh2, gW2) = res
    assert torch.equal(p1, p2) and float(o1["loss"]) == float(o2["loss"])
    assert torch.equal(o1["predicted"], o2["predicted"])
    assert torch.equal(gh1, gh2) and torch.equal(gW1, gW2)
    ref = flce_oracle(h, W, y)
    assert abs(float(o1["loss"]) - ref["loss"]) <= 2e-3 * abs(ref["loss"])
    assert np.abs(gh1.double().cpu().numpy() - ref["grad_h"]).max() <= 1e-2 * np.abs(ref["grad_h"]).max()
    assert np.abs(gW1.double().cpu().numpy() - ref["grad_W"]).max() <= 1e-2 * np.abs(ref["grad_W"]).max()


def test_pair_bounded_waits_time_out_and_context_survives(flce):
    """The test hook makes both CTAs' loaders issue nothing: the leader's MMA
    waits and both CTAs' epilogue waits give up after the limit, each CTA on
    its own clock, and both reach the closing cluster barrier, free TMEM and
    return with FLCE_ERR_TIMEOUT; the next call on the context is correct."""
    N, H, V = 256, 128, 1024
    h, W, y = _inputs(N, H, V, 73)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    flce.flce_ce_only(hd, Wd, yd, flags=flce.FLCE_FLAG_TEST_STALL | TILE256 | PAIR, timeout_ns=50_000_000)
    st = flce.flce_get_status()
    assert st & 32, st
    loss, acc = flce.flce_ce_only(hd, Wd, yd, flags=TILE256 | PAIR)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=False)
    assert abs(float(loss) - ref["loss"]) <= 2e-3 * ref["loss"]
