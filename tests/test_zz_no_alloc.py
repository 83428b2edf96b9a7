"""The CE-only entry point that allocates no device memory (flce_ce_only_noalloc).

It serves callers that cannot allocate at the point where they need the loss,
such as code running inside an allocator's callbacks or under a framework's
allocator lock. Its scratch is a fixed device array inside the library.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test. It must pass both on its own in a
fresh process and after the rest of the suite.
"""
import ctypes

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


def _call_noalloc(flce, h, W, y, **kw):
    """Straight through the C ABI (ctypes), with caller-owned outputs."""
    from linear_cross_entropy_02_gb300 import _lib
    L = _lib.lib()
    p = flce._params(h.shape[0], W.shape[1], W.shape[0], h.stride(0), W.stride(0), kw.get("softcap", 0.0),
                     kw.get("out_mult", 1.0), -100, "mean", 1.0, 0, 0, 0)
    loss = torch.full((), float("nan"), dtype=torch.float32, device=DEV)
    acc = torch.full((), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.full((), -1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    rc = L.flce_ce_only_noalloc(ctypes.byref(p), ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                ctypes.c_void_p(acc.data_ptr()), ctypes.c_void_p(st.data_ptr()), stream)
    return rc, loss, acc, st


def _oracle_check(h, W, y, loss, acc, **kw):
    """The fp64 oracle on the same inputs: loss within 2e-3 relative; the
    correct count exact up to one per valid row whose oracle top-2 gap is a
    near tie (< 1e-3 relative), where the argmax may go either way."""
    ref = flce_oracle(h.cpu(), W.cpu(), y.cpu(), need_grad_h=False, need_grad_W=False, **kw)
    assert abs(float(loss) - ref["loss"]) <= 2e-3 * abs(ref["loss"]), (float(loss), ref["loss"])
    valid = y.cpu().numpy() != -100
    slack = int(np.sum((ref["top2_gap"] < 1e-3) & valid))
    assert abs(round(float(acc) * ref["n_valid"]) - ref["correct"]) <= slack


@pytest.mark.parametrize("case", [
    dict(N=700, H=192, V=3001, seed=31),                                  # several tiles, ragged tails
    dict(N=9000, H=256, V=40000, seed=32, softcap=30.0, out_mult=0.5),    # more than one chunk
    # a Muse-sized vocabulary: its partials need more than the array at
    # 8192-row chunks, so the call falls back to 4096-row chunks (three here)
    dict(N=8500, H=64, V=202048, seed=33, softcap=30.0, out_mult=0.5),
])
def test_noalloc_matches_ce_only_on_two_calls_in_a_row(flce, case):
    N, H, V, seed = case["N"], case["H"], case["V"], case["seed"]
    kw = {k: case[k] for k in ("softcap", "out_mult") if k in case}
    results = []
    for call in range(2):
        # the second call uses other inputs, so leftovers of the first would show
        h = workloads.make_hidden(N, H, seed + call).to(DEV)
        W = workloads.make_weight(V, H, seed + call, std=0.05).to(DEV)
        y = workloads.make_labels(N, V, seed + call, 0.1).to(DEV)
        rc, loss, acc, st = _call_noalloc(flce, h, W, y, **kw)
        assert rc == 0, flce._lib.lib().flce_status_string(rc)
        ref_loss, ref_acc = flce.flce_ce_only(h, W, y, **kw)
        torch.cuda.synchronize()
        assert int(st) == 0
        assert abs(float(loss) - float(ref_loss)) <= 2e-3 * abs(float(ref_loss))
        n_valid = int((y != -100).sum())
        assert round(float(acc) * n_valid) == round(float(ref_acc) * n_valid)
        _oracle_check(h, W, y, loss, acc, **kw)
        results.append(float(loss))
    assert results[0] != results[1]


def test_noalloc_rejects_vocab_beyond_its_scratch(flce):
    from linear_cross_entropy_02_gb300 import _lib
    L = _lib.lib()
    # 20M vocab entries need more than the fixed 64 MiB even at 128-row chunks;
    # the call must fail on the host before touching any pointer
    p = flce._params(128, 8, 20_000_000, 8, 8, 0.0, 1.0, -100, "mean", 1.0, 0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)
    rc = L.flce_ce_only_noalloc(ctypes.byref(p), fake, fake, fake, fake, None, None, None)
    assert rc == _lib.FLCE_ERR_WORKSPACE
    assert L.flce_status_string(rc) == b"workspace too small"


def test_noalloc_python_wrapper(flce):
    w = workloads.WORKLOADS["tiny"]
    h, W, y = (t.to(DEV) for t in workloads.make_inputs(w))
    loss, acc, st = flce.flce_ce_only_noalloc(h, W, y)
    ref_loss, ref_acc = flce.flce_ce_only(h, W, y)
    torch.cuda.synchronize()
    assert int(st) == 0
    assert abs(float(loss) - float(ref_loss)) <= 2e-3 * abs(float(ref_loss))
    assert float(acc) == float(ref_acc)
    _oracle_check(h, W, y, loss, acc)
