"""The C ABI from a plain C99 program (tests/c_client/flce_client.c): no C++,
no torch, only include/flce.h and the CUDA runtime's C API. On the CPU the
host-side entry points; on the GPU a forward+backward through device buffers
the program allocates itself, equal bit for bit to the Python binding's call
and within tolerance of the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads
from oracle import flce_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    import __graft_entry__
    __graft_entry__.build()
    from linear_cross_entropy_02_gb300 import _lib
    pkg = os.path.dirname(_lib.LIB_PATH)
    libdir = next((d for d in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"))
                   if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    if libdir is None:
        pytest.skip("no libcudart.so next to the CUDA toolkit")
    exe = str(tmp_path_factory.mktemp("c_client") / "flce_client")
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_client", "flce_client.c"),
           "-L", pkg, "-lflce", "-L", libdir, "-lcudart", f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_host_entry_points_from_c(client):
    import linear_cross_entropy_02_gb300 as flce
    N, H, V = 32768, 7168, 129280
    r = subprocess.run([client, "host", str(N), str(H), str(V)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = r.stdout.strip().splitlines()
    kv, plain = {}, {}
    for ln in out:
        key, rest = ln.split(" ", 1)
        if "=" in rest:
            for item in rest.split():
                k, v = item.split("=", 1)
                kv[f"{key}.{k}"] = v
        elif key != "status":
            plain[key] = rest
    assert (kv["default.softcap"], kv["default.out_mult"], kv["default.ignore_index"], kv["default.reduction"],
            kv["default.grad_scale"], kv["default.chunk_rows"]) == ("0", "1", "-100", "0", "1", "0")
    assert int(kv["workspace.forward_backward"]) == flce.flce_workspace_size(N, H, V)
    assert int(kv["workspace.ce_only"]) == flce.flce_workspace_size(N, H, V, mode=flce.FLCE_MODE_CE_ONLY)
    assert 0 < int(kv["workspace.ce_only"]) < int(kv["workspace.forward_backward"])
    assert kv["workspace.bad_hidden"] == "0"                           # H % 8 != 0: invalid
    assert int(plain["no_buffers"]) == 1                               # FLCE_ERR_ARG, before any launch
    assert plain["kernel0"] == "prologue"
    status = [ln for ln in out if ln.startswith("status")]
    assert status[0] == "status 0 ok" and len(status) == 8


@pytest.mark.gpu
def test_forward_backward_from_c(client, tmp_path):
    import linear_cross_entropy_02_gb300 as flce
    N, H, V, C, T, m = 300, 136, 777, 128, 30.0, 0.5
    h = workloads.make_hidden(N, H, 81)
    W = workloads.make_weight(V, H, 81, std=0.05)
    y = workloads.make_labels(N, V, 81, 0.1)
    G0 = (np.random.default_rng(81).standard_normal((V, H)) * 1e-3).astype(np.float32)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([N, H, V, C], dtype="<i8").tobytes())
        f.write(np.array([T, m], dtype="<f4").tobytes())
        f.write(h.view(torch.int16).numpy().astype("<i2").tobytes())
        f.write(W.view(torch.int16).numpy().astype("<i2").tobytes())
        f.write(y.numpy().astype("<i8").tobytes())
        f.write(G0.astype("<f4").tobytes())
    r = subprocess.run([client, "gpu", str(inp), str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(out, "rb").read()
    o = 0
    sc = np.frombuffer(raw, "<f4", 2, o); o += 8
    codes = np.frombuffer(raw, "<i4", 2, o); o += 8
    pred = np.frombuffer(raw, "<i8", N, o); o += 8 * N
    gh = np.frombuffer(raw, "<i2", N * H, o); o += 2 * N * H
    gw = np.frombuffer(raw, "<f4", V * H, o); o += 4 * V * H
    assert o == len(raw) and list(codes) == [0, 0]

    dev = torch.device("cuda", 0)
    gW = torch.from_numpy(G0.copy()).to(dev)
    ref = flce.flce_forward_backward(h.to(dev), W.to(dev), y.to(dev), grad_W=gW, softcap=T, out_mult=m,
                                     chunk_rows=C, return_predicted=True)
    torch.cuda.synchronize()
    assert float(sc[0]) == float(ref["loss"]) and float(sc[1]) == float(ref["token_accuracy"])
    assert np.array_equal(pred, ref["predicted"].cpu().numpy())
    assert np.array_equal(gh, ref["grad_h"].cpu().view(torch.int16).numpy().reshape(-1))
    assert np.array_equal(gw, gW.cpu().numpy().reshape(-1))
    orc = flce_oracle(h, W, y, softcap=T, out_mult=m, grad_W0=G0.astype(np.float64))
    assert abs(float(sc[0]) - orc["loss"]) <= 2e-3 * abs(orc["loss"])
    gwd = gw.reshape(V, H).astype(np.float64)
    assert np.abs(gwd - orc["grad_W"]).max() <= 1e-2 * np.abs(orc["grad_W"] - G0).max()


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["vp", "vps"])
def test_vocab_parallel_from_c(client, tmp_path, mode):
    """The vocabulary-parallel entry points driven from C alone: three shards
    run in turn on buffers the C program allocates (vps: each shard keeps its
    logits between its calls, FLCE_FLAG_VP_STORED, in a workspace of its own).
    Predictions and accuracy equal the unsharded call's, the loss agrees to
    the fp32 merge order, and grad_h (summed in fp32 over the shards) and
    grad_W match the oracle."""
    import linear_cross_entropy_02_gb300 as flce
    N, H, V, C, T, m, S = 300, 136, 777, 128, 30.0, 0.5, 3
    h = workloads.make_hidden(N, H, 82)
    W = workloads.make_weight(V, H, 82, std=0.05)
    y = workloads.make_labels(N, V, 82, 0.1)
    G0 = (np.random.default_rng(82).standard_normal((V, H)) * 1e-3).astype(np.float32)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([N, H, V, C], dtype="<i8").tobytes())
        f.write(np.array([T, m], dtype="<f4").tobytes())
        f.write(h.view(torch.int16).numpy().astype("<i2").tobytes())
        f.write(W.view(torch.int16).numpy().astype("<i2").tobytes())
        f.write(y.numpy().astype("<i8").tobytes())
        f.write(G0.astype("<f4").tobytes())
    r = subprocess.run([client, mode, str(inp), str(out), str(S)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(out, "rb").read()
    o = 0
    sc = np.frombuffer(raw, "<f4", 2, o); o += 8
    codes = np.frombuffer(raw, "<i4", 2, o); o += 8
    pred = np.frombuffer(raw, "<i8", N, o); o += 8 * N
    gh = np.frombuffer(raw, "<f4", N * H, o); o += 4 * N * H
    gw = np.frombuffer(raw, "<f4", V * H, o); o += 4 * V * H
    assert o == len(raw) and list(codes) == [0, 0]

    dev = torch.device("cuda", 0)
    ref = flce.flce_forward(h.to(dev), W.to(dev), y.to(dev), softcap=T, out_mult=m, chunk_rows=C)
    torch.cuda.synchronize()
    assert np.array_equal(pred, ref["predicted"].cpu().numpy())
    assert float(sc[1]) == float(ref["token_accuracy"])
    assert abs(float(sc[0]) - float(ref["loss"])) <= 1e-6 * abs(float(ref["loss"]))
    orc = flce_oracle(h, W, y, softcap=T, out_mult=m, grad_W0=G0.astype(np.float64))
    assert np.abs(gh.reshape(N, H) - orc["grad_h"]).max() <= 1e-2 * np.abs(orc["grad_h"]).max()
    gwd = gw.reshape(V, H).astype(np.float64)
    assert np.abs(gwd - orc["grad_W"]).max() <= 1e-2 * np.abs(orc["grad_W"] - G0).max()
