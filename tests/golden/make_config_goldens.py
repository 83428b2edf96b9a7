"""Writes the oracle's full-size forward results for the four large LM-head
workloads, so the GPU tests can compare every row of those heads with the
fp64 oracle without running it for minutes on the test machine.

Run from the repository root on any CPU machine:

    python tests/golden/make_config_goldens.py [llama muse dsv3 frozen]

It imports only `oracle` and `workloads`. For each workload it draws the
seeded inputs, runs `flce_oracle` over ALL rows in fp64 (forward only: the
per-row lse, argmax and top-2 gap do not depend on gradients), and writes

  tests/golden/configs/<name>.npz   per row: lse (fp32-rounded), predicted
                                    (int32), top2_gap (fp32-rounded), near_tie
                                    (uint8: gap < 1e-3, decided in fp64) and
                                    row_loss (fp32-rounded)
  tests/golden/configs/<name>.json  loss (fp64), correct, n_valid, near-tie
                                    counts, the sha256 of the h / W / labels
                                    bytes the recipe produced, and a planted
                                    case: a seeded half of the valid rows
                                    relabelled with the oracle's own argmax,
                                    with the oracle's loss and correct count
                                    for those labels

The lse and predicted tokens of a row do not depend on its label, so the
planted case reuses them; its loss and correct count come from a second
oracle run on the planted labels. The frozen projection's CE-only and
forward + grad_h workloads share one set of inputs (seed 4), stored once as
"frozen". The test machine regenerates the inputs with the same recipe and
checks the hashes first, so a change in the random streams cannot pass as a
kernel mismatch.
"""
from __future__ import annotations

import json
import os
import platform
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from oracle import flce_oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "configs")
NEAR_TIE = 1e-3          # relative top-2 gap below which a predicted token may differ
PLANT_FRAC = 0.5
PLANT_SEED_BASE = 500

# golden name -> workload whose inputs it holds
CONFIGS = {"llama": "llama", "muse": "muse", "dsv3": "dsv3", "frozen": "frozen_ce"}
PLANTED = ("llama", "muse")


def run_one(name: str) -> dict:
    w = workloads.WORKLOADS[CONFIGS[name]]
    t0 = time.time()
    h, W, y = workloads.make_inputs(w)
    kw = dict(softcap=w.softcap, out_mult=w.out_mult, need_grad_h=False, need_grad_W=False)
    o = flce_oracle(h, W, y, **kw)
    near = o["top2_gap"] < NEAR_TIE
    valid = y.numpy() != workloads.IGNORE_INDEX
    meta = {
        "name": name, "workload": w.name, "n_rows": w.n_rows, "hidden": w.hidden, "vocab": w.vocab,
        "softcap": w.softcap, "out_mult": w.out_mult, "seed": w.seed,
        "sha256": {"h": workloads.tensor_sha256(h), "W": workloads.tensor_sha256(W),
                   "labels": workloads.tensor_sha256(y)},
        "loss": float(o["loss"]), "correct": int(o["correct"]), "n_valid": int(o["n_valid"]),
        "token_accuracy": float(o["token_accuracy"]),
        "near_tie_threshold": NEAR_TIE,
        "near_tie_rows": int(near.sum()), "near_tie_valid_rows": int((near & valid).sum()),
        "generated_by": "tests/golden/make_config_goldens.py (oracle.flce_oracle, fp64, all rows)",
        "torch": torch.__version__, "numpy": np.__version__, "machine": platform.machine(),
    }
    if name in PLANTED:
        seed = PLANT_SEED_BASE + w.seed
        yp = workloads.plant_labels(y, o["predicted"], PLANT_FRAC, seed)
        op = flce_oracle(h, W, yp, **kw)
        assert np.array_equal(op["predicted"], o["predicted"]) and np.array_equal(op["lse"], o["lse"])
        meta["planted"] = {"frac": PLANT_FRAC, "seed": seed, "sha256_labels": workloads.tensor_sha256(yp),
                           "loss": float(op["loss"]), "correct": int(op["correct"]),
                           "n_valid": int(op["n_valid"]), "token_accuracy": float(op["token_accuracy"])}
    meta["elapsed_s"] = round(time.time() - t0, 1)
    np.savez_compressed(os.path.join(OUT, f"{name}.npz"),
                        lse=o["lse"].astype(np.float32), predicted=o["predicted"].astype(np.int32),
                        top2_gap=o["top2_gap"].astype(np.float32), near_tie=near.astype(np.uint8),
                        row_loss=o["row_loss"].astype(np.float32))
    with open(os.path.join(OUT, f"{name}.json"), "w") as f:
        json.dump(meta, f, indent=1, sort_keys=True)
        f.write("\n")
    return meta


def main(argv):
    names = argv[1:] or list(CONFIGS)
    os.makedirs(OUT, exist_ok=True)
    for n in names:
        if n not in CONFIGS:
            raise SystemExit(f"unknown golden {n!r}; choose from {sorted(CONFIGS)}")
        m = run_one(n)
        print(f"{n}: loss {m['loss']:.9f} correct {m['correct']}/{m['n_valid']} "
              f"near-tie rows {m['near_tie_rows']} ({m['elapsed_s']} s)", flush=True)


if __name__ == "__main__":
    main(sys.argv)
