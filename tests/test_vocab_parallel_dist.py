"""The exchange of the vocabulary-parallel head across ranks, on CPU with gloo
(world size 2): each rank holds one vocabulary shard of W, computes its
per-row partials and its part of grad_h (here with the fp64 oracle, as the CPU
stand-in for flce_vp_forward / flce_vp_backward), and the package's exchange
helpers build the shard table, gather the partials in vocabulary order and sum
the grad_h parts. Rank 1 holds the LOWER shard, so a gather that kept rank
order instead of vocabulary order would fail. Merged, the result must equal
the unsharded oracle on every rank."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import linear_cross_entropy_02_gb300 as flce
    from oracle import flce_oracle, oracle_merge_shards, oracle_shard_grad_h, oracle_shard_partials

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(60)
        N, H, V = 40, 6, 29
        h = rng.standard_normal((N, H))
        W = rng.standard_normal((V, H))
        lab = rng.integers(0, V, N)
        lab[:4] = -100
        T, m = 3.0, 0.5
        bounds = {1: (0, 12), 0: (12, V)}[rank]          # rank 1 holds the lower ids
        v0, v1 = bounds
        offsets, order = flce.vp_shard_table(v0, v1 - v0)
        assert offsets == [0, 12, V] and order == [1, 0], (offsets, order)
        # this rank's partials for its shard, [4, N] like flce_vp_forward's
        part = oracle_shard_partials(h, W, lab, [0, v0, v1] if v0 else [0, v1], softcap=T, out_mult=m)
        k = 1 if v0 else 0
        mine = torch.tensor(np.stack([part["max"][k], part["sumexp"][k], part["argmax"][k].astype(np.float64),
                                      part["target"][k]]))
        allp = flce.vp_gather_partials(mine, order)
        assert tuple(allp.shape) == (2, 4, N)
        gathered = {"max": allp[:, 0].numpy(), "sumexp": allp[:, 1].numpy(),
                    "argmax": allp[:, 2].numpy().astype(np.int64), "target": allp[:, 3].numpy()}
        merged = oracle_merge_shards(gathered, lab, offsets)
        full = flce_oracle(h, W, lab, softcap=T, out_mult=m)
        ok_fwd = (abs(merged["loss"] - full["loss"]) <= 1e-12 * abs(full["loss"])
                  and np.array_equal(merged["predicted"], full["predicted"])
                  and np.allclose(merged["lse"], full["lse"], rtol=1e-14))
        gh = torch.tensor(oracle_shard_grad_h(h, W, lab, merged["lse"], merged["n_valid"], v0, v1, softcap=T,
                                              out_mult=m))
        flce.vp_reduce_grad_h(gh)
        ok_bwd = np.allclose(gh.numpy(), full["grad_h"], rtol=1e-10, atol=1e-14)
        q.put((rank, bool(ok_fwd), bool(ok_bwd)))
    except Exception as e:  # report at once instead of letting the parent wait out its timeout
        q.put((rank, False, False, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


def test_vocab_parallel_exchange_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, True, True), (1, True, True)]
