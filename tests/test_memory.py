"""Transient memory of a call: the library allocates nothing itself, so a
forward+backward needs no device memory beyond its inputs, its outputs and the
workspace flce_workspace_size reports; that workspace is set by the chunk size
and does not grow with the number of rows (the DeepSeek-V3 page, Memory:
chunked transients instead of the [tokens, vocab] logits)."""
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


@pytest.mark.parametrize("low_memory", [False, True])
def test_peak_memory_is_inputs_outputs_and_workspace(flce, low_memory):
    H, V, C = 512, 50000, 1024
    flags = flce.FLCE_FLAG_RECOMPUTE if low_memory else 0
    ws_sizes = []
    for N in (1024, 2048, 4096):
        h = workloads.make_hidden(N, H, 1).to(DEV)
        W = workloads.make_weight(V, H, 1).to(DEV)
        y = workloads.make_labels(N, V, 1, 0.05).to(DEV)
        gW = torch.zeros((V, H), dtype=torch.float32, device=DEV)
        flce._workspaces.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(DEV)
        base = torch.cuda.memory_allocated(DEV)
        free_before = torch.cuda.mem_get_info(DEV)[0]
        out = flce.flce_forward_backward(h, W, y, grad_W=gW, chunk_rows=C, low_memory=low_memory)
        torch.cuda.synchronize()
        assert flce.flce_get_status() == 0
        peak = torch.cuda.max_memory_allocated(DEV) - base
        ws = flce.flce_workspace_size(N, H, V, chunk_rows=C, flags=flags)
        ws_sizes.append(ws)
        outputs = N * H * 2 + 3 * 512          # grad_h (bf16) + the scalars, allocator-rounded
        assert peak <= ws + outputs + (2 << 20), (peak, ws, outputs)
        # nothing outside torch's allocator: the device's free memory fell by no
        # more than what torch reserved
        reserved = torch.cuda.memory_reserved(DEV)
        free_after = torch.cuda.mem_get_info(DEV)[0]
        assert free_before - free_after <= reserved + (256 << 20)   # slack: module loading
        del out
    assert len(set(ws_sizes)) == 1                  # independent of N at a fixed chunk size
    # and far below a [N, V] fp32 logits tensor at the largest N
    assert ws_sizes[0] < 4096 * V * 4
