"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle on
the same seeded inputs, element by element, at sizes that span several tiles
and ragged tails. Tolerances (the contract of this library):
  loss: relative error <= 2e-3
  grad_h, grad_W: max-abs error <= 1e-2 * max|ref|
  predicted_tokens: exact on every row whose oracle top-2 gap is >= 1e-3 relative;
                    near-tie rows are counted and reported
  token_accuracy: exact correct count, up to near-tie rows whose label is one of
                  the two candidates
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle

pytestmark = pytest.mark.gpu

LOSS_RTOL = 2e-3
GRAD_TOL = 1e-2
GAP = 1e-3


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


DEV = torch.device("cuda", 0)


def _inputs(N, H, V, seed, ign=0.1, W_scale=0.02, labels="uniform"):
    h = workloads.make_hidden(N, H, seed)
    W = workloads.make_weight(V, H, seed, std=W_scale)
    y = workloads.make_labels(N, V, seed, ign, labels)
    return h, W, y


def check_against_oracle(out, ref, labels, *, grad_W0=None, what=""):
    lab = labels.numpy()
    valid = lab != -100
    loss = float(out["loss"])
    if ref["n_valid"] == 0:
        assert loss == 0.0, what
    else:
        assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"]), (what, loss, ref["loss"])
    report = {}
    if out.get("predicted") is not None:
        pred = out["predicted"].reshape(-1).cpu().numpy()
        near = ref["top2_gap"] < GAP
        bad = (pred != ref["predicted"]) & ~near
        assert not bad.any(), (what, "argmax mismatch on rows", np.nonzero(bad)[0][:10])
        report["near_tie_rows"] = int(near.sum())
        # the accuracy must be the GPU's own argmax count, and may differ from the
        # oracle's count only on near-tie rows where one of the two is the label
        n_valid = int(valid.sum())
        acc = float(out["token_accuracy"])
        gpu_correct = int(np.sum(valid & (pred == lab)))
        if n_valid:
            assert round(acc * n_valid) == gpu_correct, (what, acc, gpu_correct)
        diff_rows = valid & (pred != ref["predicted"]) & ((pred == lab) | (ref["predicted"] == lab))
        assert abs(gpu_correct - ref["correct"]) <= int(diff_rows.sum()), what
    else:
        n_valid = ref["n_valid"]
        if n_valid:
            acc = float(out["token_accuracy"])
            assert round(acc * n_valid) == ref["correct"], (what, acc * n_valid, ref["correct"])
    if out.get("grad_h") is not None and ref.get("grad_h") is not None:
        gh = out["grad_h"].reshape(ref["grad_h"].shape).float().cpu().numpy()
        scale = np.abs(ref["grad_h"]).max()
        err = np.abs(gh - ref["grad_h"]).max()
        if scale == 0:
            assert err == 0, what
        else:
            assert err <= GRAD_TOL * scale, (what, "grad_h", err, scale)
        report["grad_h_err"] = float(err / max(scale, 1e-300))
    if out.get("grad_W") is not None and ref.get("grad_W") is not None:
        gw = out["grad_W"].cpu().double().numpy()
        delta_ref = ref["grad_W"] - (0.0 if grad_W0 is None else grad_W0)
        scale = np.abs(delta_ref).max()
        err = np.abs(gw - ref["grad_W"]).max()
        assert err <= GRAD_TOL * max(scale, 1e-30), (what, "grad_W", err, scale)
        report["grad_W_err"] = float(err / max(scale, 1e-300))
    return report


def run_fwd_bwd(flce, h, W, y, *, softcap=0.0, out_mult=1.0, grad_W0=None, reduction="mean",
                grad_scale=1.0, frozen=False, chunk_rows=0, flags=0, need_grad_h=True):
    gW = None
    if not frozen:
        gW = (torch.zeros(W.shape, dtype=torch.float32) if grad_W0 is None
              else torch.from_numpy(grad_W0).float()).to(DEV)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, need_grad_h=need_grad_h,
                                     softcap=softcap, out_mult=out_mult, reduction=reduction,
                                     grad_scale=grad_scale, return_predicted=True, chunk_rows=chunk_rows,
                                     flags=flags, vocab_slab=512 if flags & 8 else 0)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    return out


# 0: tcgen05 GEMMs on 256 x 256 CTA tiles, backward operands read in place as
#    MN-major tiles (the product path)
# 1: debug fp32-FMA GEMMs (FLCE_FLAG_SIMT_GEMM)
# 4: tcgen05 GEMMs fed explicit transposes, all operands K-major (FLCE_FLAG_KMAJOR_BWD)
# 8: low-memory recompute backward (FLCE_FLAG_RECOMPUTE), vocab slabs of 512 columns so
#    the shapes below span several slabs and a ragged last slab
# 16: 128 x 256 CTA tiles with two accumulators everywhere (FLCE_FLAG_TILE128)
# 32: 256 x 256 CTA tiles everywhere (FLCE_FLAG_TILE256; by default small GEMMs
#     such as these take 128-row tiles); 24 and 40: each with the recompute backward
PATHS = [0, 1, 4, 8, 16, 24, 32, 40]


@pytest.mark.parametrize("flags", PATHS)
def test_tiny_head_full(flce, flags):
    w = workloads.WORKLOADS["tiny"]
    h, W, y = workloads.make_inputs(w)
    G0 = np.random.default_rng(0).standard_normal((w.vocab, w.hidden)) * 1e-4
    G0 = G0.astype(np.float32).astype(np.float64)
    out = run_fwd_bwd(flce, h, W, y, grad_W0=G0, flags=flags)
    ref = flce_oracle(h, W, y, grad_W0=G0)
    rep = check_against_oracle(out, ref, y, grad_W0=G0, what=f"tiny flags={flags}")
    print("tiny", flags, rep)


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("case", [
    dict(N=300, H=192, V=1000, chunk_rows=128),             # ragged rows, ragged vocab tile, 3 chunks
    dict(N=129, H=64, V=4100, chunk_rows=0),                 # H = one K slice, V tail of 4 columns
    dict(N=513, H=136, V=777, chunk_rows=256, softcap=30.0, out_mult=0.5),  # H % 64 != 0, softcap, m
    dict(N=256, H=256, V=2048, softcap=2.0, out_mult=0.5, reduction="sum", grad_scale=0.75),
    # chunks of 768 and 332 rows: three 256-row units, then two (the second
    # ending 180 rows past the data); V = 1500 gives six vocab units for grad_W
    dict(N=1100, H=192, V=1500, chunk_rows=768),
])
def test_edge_shapes(flce, flags, case):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    h, W, y = _inputs(N, H, V, seed=N + V, W_scale=0.05)
    G0 = (np.random.default_rng(1).standard_normal((V, H)) * 1e-3).astype(np.float32).astype(np.float64)
    out = run_fwd_bwd(flce, h, W, y, grad_W0=G0, flags=flags, **c)
    ref = flce_oracle(h, W, y, grad_W0=G0, softcap=c.get("softcap", 0.0), out_mult=c.get("out_mult", 1.0),
                      reduction=c.get("reduction", "mean"), grad_scale=c.get("grad_scale", 1.0))
    rep = check_against_oracle(out, ref, y, grad_W0=G0, what=f"{case} flags={flags}")
    print(case, flags, rep)


@pytest.mark.parametrize("flags", PATHS)
def test_zero_weight_gives_ln_v(flce, flags):
    N, H, V = 200, 128, 5000
    h, _, y = _inputs(N, H, V, seed=3)
    W = torch.zeros((V, H), dtype=torch.bfloat16)
    out = run_fwd_bwd(flce, h, W, y, softcap=30.0, flags=flags)
    assert abs(float(out["loss"]) - np.log(V)) <= 1e-5 * np.log(V)
    assert torch.all(out["grad_h"] == 0)
    assert torch.all(out["predicted"].cpu() == 0)      # all logits tie: lowest index
    ref = flce_oracle(h, W, y, softcap=30.0)
    check_against_oracle(out, ref, y, what="W=0")


@pytest.mark.parametrize("flags", PATHS)
def test_all_ignored(flce, flags):
    N, H, V = 160, 64, 700
    h, W, _ = _inputs(N, H, V, seed=4)
    y = torch.full((N,), -100, dtype=torch.int64)
    G0 = np.full((V, H), 0.25)
    out = run_fwd_bwd(flce, h, W, y, grad_W0=G0, flags=flags)
    assert float(out["loss"]) == 0.0 and float(out["token_accuracy"]) == 0.0
    assert torch.all(out["grad_h"] == 0)
    assert torch.all(out["grad_W"] == 0.25)


def test_planted_accuracy(flce):
    N, H, V = 384, 128, 3000
    h, W, y = _inputs(N, H, V, seed=5, W_scale=0.1)
    pred = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=False)["predicted"]
    valid = np.nonzero(y.numpy() != -100)[0]
    plant = np.random.default_rng(2).choice(valid, size=len(valid) // 2, replace=False)
    y2 = y.clone()
    y2[plant] = torch.from_numpy(pred[plant])
    out = run_fwd_bwd(flce, h, W, y2)
    ref = flce_oracle(h, W, y2)
    assert ref["token_accuracy"] >= 0.5
    check_against_oracle(out, ref, y2, what="planted")


@pytest.mark.parametrize("flags", [0, 8, 16, 32])
def test_frozen_weight_and_no_grad_h(flce, flags):
    N, H, V = 256, 128, 2000
    h, W, y = _inputs(N, H, V, seed=6)
    out = run_fwd_bwd(flce, h, W, y, frozen=True, flags=flags)
    assert out["grad_W"] is None
    ref = flce_oracle(h, W, y, need_grad_W=False)
    check_against_oracle(out, ref, y, what="frozen")
    out2 = run_fwd_bwd(flce, h, W, y, need_grad_h=False, flags=flags)
    assert out2["grad_h"] is None
    check_against_oracle(out2, flce_oracle(h, W, y), y, what="grad_W only")


def test_forward_and_ce_only_agree(flce):
    N, H, V = 400, 192, 3333
    h, W, y = _inputs(N, H, V, seed=7)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    f = flce.flce_forward(hd, Wd, yd, return_lse=True, softcap=5.0, out_mult=0.5)
    loss_ce, acc_ce = flce.flce_ce_only(hd, Wd, yd, softcap=5.0, out_mult=0.5)
    fb = flce.flce_forward_backward(hd, Wd, yd, grad_W=torch.zeros(W.shape, device=DEV), softcap=5.0,
                                    out_mult=0.5, return_predicted=True)
    torch.cuda.synchronize()
    ref = flce_oracle(h, W, y, softcap=5.0, out_mult=0.5, need_grad_h=False, need_grad_W=False)
    assert float(loss_ce) == float(f["loss"]) == float(fb["loss"])
    assert float(acc_ce) == float(f["token_accuracy"]) == float(fb["token_accuracy"])
    lse = f["lse"].cpu().double().numpy()
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * np.abs(ref["lse"]).max()
    assert torch.equal(f["predicted"], fb["predicted"])
    check_against_oracle({"loss": loss_ce, "token_accuracy": acc_ce}, ref, y, what="ce_only")


def test_ce_only_touches_no_gradient_buffer_and_launches_less(flce):
    N, H, V = 300, 128, 1500
    h, W, y = _inputs(N, H, V, seed=8)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    canary = torch.full((V, H), 7.0, device=DEV)
    n0 = flce.flce_launch_count()
    flce.flce_ce_only(hd, Wd, yd)
    n_ce = flce.flce_launch_count() - n0
    n0 = flce.flce_launch_count()
    flce.flce_forward(hd, Wd, yd)
    n_fwd = flce.flce_launch_count() - n0
    n0 = flce.flce_launch_count()
    flce.flce_forward_backward(hd, Wd, yd, grad_W=torch.zeros(W.shape, device=DEV))
    n_bwd = flce.flce_launch_count() - n0
    torch.cuda.synchronize()
    assert torch.all(canary == 7.0)
    assert n_ce <= n_fwd < n_bwd


def test_invalid_label_sets_status_without_fault(flce):
    N, H, V = 128, 64, 500
    h, W, y = _inputs(N, H, V, seed=9)
    y[5] = V + 3
    y[9] = -7
    flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV))
    assert flce.flce_get_status() & 16
    # the next call on the same context is clean
    y[5], y[9] = 0, 1
    flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV))
    assert flce.flce_get_status() == 0


def test_bounded_wait_times_out_and_context_survives(flce):
    """The test hook makes the forward GEMM's loader issue nothing; the MMA and
    epilogue waits must give up after the limit, set FLCE_ERR_TIMEOUT, free
    TMEM and return, and the next call must run normally."""
    N, H, V = 256, 128, 1024
    h, W, y = _inputs(N, H, V, seed=10)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    flce.flce_ce_only(hd, Wd, yd, flags=flce.FLCE_FLAG_TEST_STALL, timeout_ns=50_000_000)
    st = flce.flce_get_status()
    assert st & 32, st
    loss, acc = flce.flce_ce_only(hd, Wd, yd)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, need_grad_h=False, need_grad_W=False)
    assert abs(float(loss) - ref["loss"]) <= LOSS_RTOL * ref["loss"]


def test_proposal_rows_shape_restored(flce):
    """[B, k, S, H] proposal rows are flattened for the frozen projection and
    per-row outputs come back as [B, k, S] (SpecForge DSpine PR, Changes)."""
    B, k, S, H, V = 2, 3, 40, 64, 900
    h, W, y = _inputs(B * k * S, H, V, seed=11)
    h4 = h.view(B, k, S, H).to(DEV)
    y3 = y.view(B, k, S).to(DEV)
    out = flce.flce_forward_backward(h4, W.to(DEV), y3, grad_W=None, return_predicted=True)
    torch.cuda.synchronize()
    assert out["grad_h"].shape == (B, k, S, H) and out["predicted"].shape == (B, k, S)
    ref = flce_oracle(h, W, y, need_grad_W=False)
    check_against_oracle({"loss": out["loss"], "token_accuracy": out["token_accuracy"],
                          "predicted": out["predicted"], "grad_h": out["grad_h"]}, ref, y, what="4d")


def test_zipf_labels_and_row_sums(flce):
    """Zipf labels (the DeepSeek-V3-shaped workload's recipe); with no softcap
    the columns of grad_W sum to zero over the vocabulary."""
    N, H, V = 512, 256, 6000
    h = workloads.make_hidden(N, H, 12)
    W = workloads.make_weight(V, H, 12)
    y = workloads.make_labels(N, V, 12, 0.03, "zipf", 1.1)
    out = run_fwd_bwd(flce, h, W, y)
    ref = flce_oracle(h, W, y)
    check_against_oracle(out, ref, y, what="zipf")
    # up to the bf16 rounding of dz: |sum_j gW_jk| <= 2^-8 / n_valid * sum_{valid i} |h_ik|
    col = out["grad_W"].double().sum(dim=0).abs()
    valid = y != -100
    bound = 2.0 ** -8 / int(valid.sum()) * h[valid].double().abs().sum(0).to(DEV)
    assert torch.all(col <= bound)


@pytest.mark.parametrize("flags", [0, 8, 16, 32])
@pytest.mark.parametrize("case", [
    dict(N=5, H=64, V=100),                                   # one partial row tile, V < one vocab tile
    dict(N=130, H=128, V=257, ignore_index=-1),               # custom ignore index, one column past a tile
    dict(N=200, H=64, V=1000, out_mult=-0.5, softcap=3.0),    # negative multiplier: the argmax flips
    dict(N=70, H=8, V=300),                                   # H = 8: one 16-byte row per operand row
    dict(N=40, H=64, V=1),                                    # one class: loss 0, every gradient 0
])
def test_small_and_unusual_heads(flce, flags, case):
    c = dict(case)
    N, H, V = c.pop("N"), c.pop("H"), c.pop("V")
    ign = c.pop("ignore_index", -100)
    h, W, y = _inputs(N, H, V, seed=N * 7 + V, W_scale=0.1)
    y = torch.where(y == -100, torch.full_like(y, ign), y)
    gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    out = flce.flce_forward_backward(h.to(DEV), W.to(DEV), y.to(DEV), grad_W=gW, ignore_index=ign,
                                     return_predicted=True, flags=flags, vocab_slab=256 if flags & 8 else 0, **c)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    ref = flce_oracle(h, W, y, ignore_index=ign, softcap=c.get("softcap", 0.0), out_mult=c.get("out_mult", 1.0))
    lab = torch.where(y == ign, torch.full_like(y, -100), y)       # the checker's ignored-row marker
    check_against_oracle(out, ref, lab, what=f"{case} flags={flags}")


def test_strided_hidden_rows(flce):
    """h with a row stride larger than H (a view into a wider buffer) is read in place."""
    N, H, V = 300, 128, 2000
    big, W, y = _inputs(N, 192, V, seed=13)
    h = big[:, :H]
    W = W[:, :H].contiguous()
    assert h.stride(0) == 192
    gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    out = flce.flce_forward_backward(big.to(DEV)[:, :H], W.to(DEV), y.to(DEV), grad_W=gW, return_predicted=True)
    torch.cuda.synchronize()
    check_against_oracle(out, flce_oracle(h, W, y), y, what="strided h")


@pytest.mark.parametrize("flags", [0, 8, 32])
def test_strided_weight_rows(flce, flags):
    """W with a row stride larger than H (the vocabulary rows of a wider
    matrix) is read in place by the forward GEMM (K-major) and by grad_h
    (MN-major), and by the recompute path's slabs."""
    N, H, V = 300, 128, 2000
    h, Wbig, y = _inputs(N, H + 64, V, seed=14, W_scale=0.05)
    h = h[:, :H].contiguous()
    W = Wbig[:, :H]
    assert W.stride(0) == H + 64
    Wd = Wbig.to(DEV)[:, :H]
    gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    out = flce.flce_forward_backward(h.to(DEV), Wd, y.to(DEV), grad_W=gW, return_predicted=True, flags=flags,
                                     chunk_rows=128, vocab_slab=512 if flags & 8 else 0)
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
    check_against_oracle(out, flce_oracle(h, W.contiguous(), y), y, what=f"strided W flags={flags}")


@pytest.mark.parametrize("flags", [0, 1])
def test_exact_tie_across_vocab_tiles_keeps_lowest_index(flce, flags):
    """Two identical rows of W in different 256-column vocab tiles (and chunks of
    the statistics) that dominate every row's logits: the capped logits tie
    bit for bit, and the argmax must be the lower index (the reading of the
    tie-break), both within the forward GEMM's tile walk and in the merge."""
    N, H, V = 96, 128, 1500
    j1, j2 = 300, 1210
    h = workloads.make_hidden(N, H, 40).abs()          # positive rows
    W = workloads.make_weight(V, H, 40)
    W[j1] = 0.5
    W[j2] = 0.5
    y = workloads.make_labels(N, V, 40, 0.1)
    y[:10] = j2                                         # labelled with the tied twin: counted as wrong
    out = run_fwd_bwd(flce, h, W, y, flags=flags)
    pred = out["predicted"].cpu()
    assert torch.all(pred == j1)
    valid = (y != -100)
    assert round(float(out["token_accuracy"]) * int(valid.sum())) == int(((y == j1) & valid).sum())


def test_empty_batch(flce):
    """No rows: the loss and accuracy are 0 (no valid rows), the per-row outputs
    are empty, grad_W is left as it was, and the call launches only the
    prologue and the finish kernels."""
    H, V = 128, 1000
    h = torch.zeros((0, H), dtype=torch.bfloat16, device=DEV)
    W = workloads.make_weight(V, H, 1).to(DEV)
    y = torch.zeros((0,), dtype=torch.int64, device=DEV)
    gW = torch.full((V, H), 0.5, dtype=torch.float32, device=DEV)
    n0 = flce.flce_launch_count()
    out = flce.flce_forward_backward(h, W, y, grad_W=gW, return_predicted=True)
    torch.cuda.synchronize()
    assert flce.flce_launch_count() - n0 == 2
    assert flce.flce_get_status() == 0
    assert float(out["loss"]) == 0.0 and float(out["token_accuracy"]) == 0.0
    assert out["grad_h"].shape == (0, H) and out["predicted"].shape == (0,)
    assert torch.all(gW == 0.5)
    f = flce.flce_forward(h, W, y, return_lse=True)
    loss, acc = flce.flce_ce_only(h, W, y)
    ce = flce.flce_cross_entropy(torch.zeros((0, V), dtype=torch.bfloat16, device=DEV), y, reduction="none")
    torch.cuda.synchronize()
    assert float(f["loss"]) == 0.0 and f["lse"].shape == (0,)
    assert float(loss) == 0.0 and float(acc) == 0.0
    assert float(ce["loss"]) == 0.0 and ce["row_loss"].shape == (0,) and ce["grad_logits"].shape == (0, V)


@pytest.mark.parametrize("flags", [0, 8, 16, 32, 40])
def test_guard_bands_around_every_output_and_the_workspace(flce, flags):
    """Through the C ABI with caller-made buffers: every output and the
    workspace sit between guard bands filled with a sentinel, on a ragged
    shape (several chunks, a partial vocab tile, H not a multiple of 64). No
    kernel writes outside the bytes it owns, and the results still match the
    oracle. On 256-row tiles the 300 rows are one chunk of two 256-row units,
    the second ending 212 rows past the data."""
    import ctypes
    from linear_cross_entropy_02_gb300 import _lib
    L = _lib.lib()
    N, H, V, C = 300, 136, 777, (384 if flags & 32 else 128)
    h, W, y = _inputs(N, H, V, seed=44, W_scale=0.05)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    G = 4096                                            # guard elements on each side

    def guarded(n, dtype, fill):
        buf = torch.full((n + 2 * G,), fill, dtype=dtype, device=DEV)
        return buf, buf[G:G + n]

    p = _lib.FlceParams()
    L.flce_default_params(ctypes.byref(p))
    p.n_rows, p.hidden, p.vocab, p.ld_h, p.ld_w, p.chunk_rows, p.flags = N, H, V, H, H, C, flags
    p.vocab_slab = 256 if flags & 8 else 0
    ws_bytes = L.flce_workspace_size(ctypes.byref(p), _lib.FLCE_MODE_FORWARD_BACKWARD, 1, 1)
    ws_buf, ws = guarded(ws_bytes, torch.uint8, 0xA5)
    gh_buf, gh = guarded(N * H, torch.bfloat16, -3.0)
    gw_buf, gw = guarded(V * H, torch.float32, 0.0)
    gw.fill_(0.0)
    gw_buf[:G].fill_(-7.0)
    gw_buf[G + V * H:].fill_(-7.0)
    pr_buf, pr = guarded(N, torch.int64, -12345)
    sc_buf, sc = guarded(2, torch.float32, -9.0)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = L.flce_forward_backward(ctypes.byref(p), ptr(hd), ptr(Wd), ptr(yd), ptr(sc[0:1]), ptr(sc[1:2]), ptr(pr),
                                 ptr(gh), ptr(gw), ptr(ws), ws_bytes,
                                 ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    st = ctypes.c_int32(-1)
    assert L.flce_get_status(ptr(ws), ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream),
                             ctypes.byref(st)) == 0 and st.value == 0
    for name, buf, n, fill in (("workspace", ws_buf, ws_bytes, 0xA5), ("grad_h", gh_buf, N * H, -3.0),
                               ("grad_W", gw_buf, V * H, -7.0), ("predicted", pr_buf, N, -12345),
                               ("scalars", sc_buf, 2, -9.0)):
        assert torch.all(buf[:G] == fill) and torch.all(buf[G + n:] == fill), name
    out = {"loss": sc[0], "token_accuracy": sc[1], "predicted": pr, "grad_h": gh.view(N, H),
           "grad_W": gw.view(V, H)}
    ref = flce_oracle(h, W, y)
    check_against_oracle(out, ref, y, what=f"guard bands flags={flags}")


@pytest.mark.parametrize("flags", [0, 32])
def test_last_vocab_column_and_large_logits(flce, flags):
    """Labels and argmax on the last vocabulary column (inside a partial vocab
    tile), and logits of several hundred in magnitude: the max-subtracted sums
    stay finite and match the oracle."""
    N, H, V = 260, 128, 777
    h, W, _ = _inputs(N, H, V, seed=51, W_scale=0.05)
    W = W.float()
    W[V - 1] = h.float()[: N].mean(0) * 4.0          # pushes column V-1 to the top for many rows
    W = (W * 60.0).to(torch.bfloat16)                 # logits of O(100s)
    y = torch.full((N,), V - 1, dtype=torch.int64)
    y[::3] = torch.arange(0, N, 3) % V
    y[5] = -100
    out = run_fwd_bwd(flce, h, W, y, flags=flags)
    assert torch.isfinite(out["loss"]).item() and torch.isfinite(out["grad_h"].float()).all()
    assert torch.isfinite(out["grad_W"]).all()
    ref = flce_oracle(h, W, y)
    assert np.abs(ref["lse"]).max() > 100.0
    assert int((out["predicted"].cpu() == V - 1).sum()) > 0
    check_against_oracle(out, ref, y, what=f"large logits flags={flags}")


def _fuzz_cases(n=64, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        cases.append(dict(
            N=int(rng.integers(1, 700)), H=int(8 * rng.integers(1, 40)), V=int(rng.integers(2, 3000)),
            softcap=float(rng.choice([0.0, 0.0, 1.5, 30.0])), out_mult=float(rng.choice([1.0, 0.5, -0.75, 2.0])),
            chunk_rows=int(rng.choice([0, 128, 256, 384])), flags=int(rng.choice([0, 8, 16, 32, 40])),
            reduction=str(rng.choice(["mean", "sum"])), ign=float(rng.choice([0.0, 0.1, 0.5])), seed=i))
    return cases


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"N{c['N']}-H{c['H']}-V{c['V']}-f{c['flags']}")
def test_fuzzed_shapes_and_options(flce, case):
    """Seeded random shapes (any N, H a multiple of 8, any V), softcaps,
    multipliers, chunk sizes, reductions, ignore fractions and GEMM paths,
    each against the oracle in full."""
    c = dict(case)
    N, H, V, flags, ign, seed = c.pop("N"), c.pop("H"), c.pop("V"), c.pop("flags"), c.pop("ign"), c.pop("seed")
    h, W, y = _inputs(N, H, V, seed=1000 + seed, ign=ign, W_scale=0.08)
    G0 = (np.random.default_rng(seed).standard_normal((V, H)) * 1e-3).astype(np.float32).astype(np.float64)
    out = run_fwd_bwd(flce, h, W, y, grad_W0=G0, flags=flags, **c)
    ref = flce_oracle(h, W, y, grad_W0=G0, softcap=c["softcap"], out_mult=c["out_mult"], reduction=c["reduction"])
    check_against_oracle(out, ref, y, grad_W0=G0, what=f"fuzz {case}")


def test_non_finite_rows_are_flagged_without_fault(flce):
    """A NaN in one row of h and an inf in another: those rows' log-sum-exp is
    not finite and the status word gets FLCE_ERR_NONFINITE; with both rows
    ignored the loss over the other rows is still the oracle's. A NaN in one
    vocabulary row of W reaches every row's sum of exponentials, in a vocab
    shard too. The next clean call reports 0."""
    N, H, V = 300, 64, 2000
    h, W, y = _inputs(N, H, V, seed=77)
    h[7, 3] = float("nan")
    h[200, 5] = float("inf")
    y[7] = -100
    y[200] = -100
    f = flce.flce_forward(h.to(DEV), W.to(DEV), y.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    assert flce.flce_get_status() & flce._lib.FLCE_ERR_NONFINITE
    lse = f["lse"].cpu()
    assert not torch.isfinite(lse[7]) and torch.isfinite(lse[[0, 8, 199, 201]]).all()
    pred = f["predicted"].cpu()
    assert pred[7] == -1 and pred[200] == -1 and (pred[[0, 8, 199, 201]] >= 0).all()
    keep = torch.ones(N, dtype=torch.bool)
    keep[[7, 200]] = False
    ref = flce_oracle(h[keep], W, y[keep], need_grad_h=False, need_grad_W=False)
    assert abs(float(f["loss"]) - ref["loss"]) <= LOSS_RTOL * ref["loss"]
    W2 = W.clone()
    W2[1500, 0] = float("nan")
    part = flce.flce_vp_forward(h.to(DEV), W2[1024:].to(DEV), y.to(DEV), 1024, V)
    torch.cuda.synchronize()
    assert flce.flce_get_status() & flce._lib.FLCE_ERR_NONFINITE
    h2, _, _ = _inputs(N, H, V, seed=78)
    flce.flce_forward(h2.to(DEV), W.to(DEV), y.to(DEV))
    torch.cuda.synchronize()
    assert flce.flce_get_status() == 0
