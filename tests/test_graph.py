"""The fused path is stream-ordered with no host synchronisation and no
allocation inside the library, so a forward+backward can be captured in a CUDA
graph once and replayed; replays match an uncaptured call. Calls on two
streams use separate workspaces."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def flce():
    import __graft_entry__
    __graft_entry__.build()
    import linear_cross_entropy_02_gb300 as m
    return m


def test_cuda_graph_capture_and_replay(flce):
    N, H, V = 1024, 256, 20000
    h = workloads.make_hidden(N, H, 21).to(DEV)
    W = workloads.make_weight(V, H, 21).to(DEV)
    y = workloads.make_labels(N, V, 21, 0.05).to(DEV)
    ref_gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    ref = flce.flce_forward_backward(h, W, y, grad_W=ref_gW, softcap=30.0, out_mult=0.5, chunk_rows=384)
    torch.cuda.synchronize()

    gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):                       # warm-up on the capture stream (workspace cached)
        flce.flce_forward_backward(h, W, y, grad_W=gW, softcap=30.0, out_mult=0.5, chunk_rows=384)
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = flce.flce_forward_backward(h, W, y, grad_W=gW, softcap=30.0, out_mult=0.5, chunk_rows=384)
    for _ in range(2):
        gW.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert float(out["loss"]) == float(ref["loss"])
        assert float(out["token_accuracy"]) == float(ref["token_accuracy"])
        assert torch.equal(out["grad_h"], ref["grad_h"])
        assert torch.equal(gW, ref_gW)              # the same launches, so the same sums


def test_two_streams_use_separate_workspaces(flce):
    N, H, V = 512, 128, 5000
    hs = [workloads.make_hidden(N, H, 30 + i).to(DEV) for i in range(2)]
    W = workloads.make_weight(V, H, 30).to(DEV)
    y = workloads.make_labels(N, V, 30, 0.05).to(DEV)
    refs = [float(flce.flce_ce_only(h, W, y)[0]) for h in hs]
    streams = [torch.cuda.Stream(DEV) for _ in range(2)]
    outs = []
    for h, st in zip(hs, streams):
        st.wait_stream(torch.cuda.current_stream(DEV))
        with torch.cuda.stream(st):
            outs.append(flce.flce_ce_only(h, W, y)[0])
    torch.cuda.synchronize()
    assert [float(o) for o in outs] == refs


@pytest.mark.parametrize("stored", [False, True], ids=["recompute", "kept_logits"])
def test_vocab_parallel_step_on_cta_pairs_captured_and_replayed(flce, stored):
    """Two vocab shards' forwards, the gather (a stack), the two backwards and
    the rounding of grad_h, all on CTA-pair GEMMs, captured once in a CUDA graph
    and replayed: the same bits as the uncaptured step. kept_logits: each shard
    keeps its logits between its calls, in a workspace allocated beforehand."""
    N, H, V = 768, 256, 9000
    offs = [0, 4000, V]
    h = workloads.make_hidden(N, H, 22).to(DEV)
    W = workloads.make_weight(V, H, 22).to(DEV)
    y = workloads.make_labels(N, V, 22, 0.05).to(DEV)
    flags = flce.FLCE_FLAG_TILE256 | flce.FLCE_FLAG_CTA_PAIR | (flce.FLCE_FLAG_VP_STORED if stored else 0)
    gh32 = torch.zeros((N, H), dtype=torch.float32, device=DEV)
    gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
    wss = [flce.flce_vp_workspace(h, W[offs[k]:offs[k + 1]], keep_logits=True) if stored else None
           for k in range(2)]

    def step():
        parts = [flce.flce_vp_forward(h, W[offs[k]:offs[k + 1]], y, offs[k], V, softcap=30.0, out_mult=0.5,
                                      flags=flags, workspace=wss[k]) for k in range(2)]
        allp = torch.stack(parts)
        gh32.zero_()
        out = None
        for k in range(2):
            out = flce.flce_vp_backward(h, W[offs[k]:offs[k + 1]], y, allp, offs, offs[k], V, grad_h_partial=gh32,
                                        grad_W=gW[offs[k]:offs[k + 1]], softcap=30.0, out_mult=0.5, flags=flags,
                                        vocab_slab=2048, workspace=wss[k])
        return out, flce.flce_scale_gradient(gh32, None, out_dtype=torch.bfloat16)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        ref, ref_gh = step()                         # uncaptured, also the warm-up of the workspace
        s.synchronize()
        ref_gW = gW.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out, gh = step()
    for _ in range(2):
        gW.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert float(out["loss"]) == float(ref["loss"]) and torch.equal(out["predicted"], ref["predicted"])
        assert torch.equal(gh, ref_gh) and torch.equal(gW, ref_gW)


def test_two_host_threads_on_two_streams(flce):
    """Two host threads, each on its own stream (and so its own cached
    workspace), call the library at once: every result equals the serial one
    bit for bit, and the status stays 0."""
    import threading
    N, H, V = 600, 192, 7000
    ins = []
    for i in range(2):
        ins.append((workloads.make_hidden(N, H, 40 + i).to(DEV), workloads.make_weight(V, H, 40 + i).to(DEV),
                    workloads.make_labels(N, V, 40 + i, 0.05).to(DEV)))
    refs = []
    for h, W, y in ins:
        o = flce.flce_forward_backward(h, W, y, return_predicted=True, softcap=30.0)
        torch.cuda.synchronize()
        refs.append((float(o["loss"]), o["predicted"].clone(), o["grad_h"].clone()))
    results = [None, None]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(DEV)
            st = torch.cuda.Stream(DEV)
            h, W, y = ins[i]
            st.wait_stream(torch.cuda.default_stream(DEV))
            outs = []
            with torch.cuda.stream(st):
                for _ in range(5):
                    o = flce.flce_forward_backward(h, W, y, return_predicted=True, softcap=30.0)
                    outs.append((o["loss"], o["predicted"], o["grad_h"]))
                st.synchronize()
                assert flce.flce_get_status() == 0
            results[i] = outs
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for i in range(2):
        for loss, pred, gh in results[i]:
            assert float(loss) == refs[i][0]
            assert torch.equal(pred, refs[i][1]) and torch.equal(gh, refs[i][2])
