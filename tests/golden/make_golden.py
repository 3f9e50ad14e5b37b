"""Write the stored oracle outputs under tests/golden/.

Calls only the oracle and the seeded input generator; no value here comes from
the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py            # every file
    python tests/golden/make_golden.py pad2048    # one of: tiny, pad2048, batched

Files (gzip-compressed text where large; np.loadtxt reads both):
  tiny_actions.txt                 2-layer fp32 tiny case, seed 0, 2 Euler steps: [16, 8]
  pi05_pad2048_actions.txt.gz      Pi0.5-shaped expert, one request of 1621..1634 valid
                                   prefix rows (the 2048-padded workload; padding does not
                                   change the oracle's result), 10 Euler steps, seeds 0..4:
                                   [5 * 50, 32], seed-major
  pi05_b16_ragged_actions.txt.gz   Pi0.5-shaped expert, 16 requests of 600..2048 valid rows,
                                   10 Euler steps, seeds 0..4: [5 * 16 * 50, 32], seed-major
                                   then request-major
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from flow_matching_action_gb300 import synth  # noqa: E402
from oracle import ae_oracle  # noqa: E402

SEEDS = (0, 1, 2, 3, 4)


def _run(wl, w):
    return ae_oracle.sample(wl.dims, w, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise, wl.n_steps)


def tiny():
    wl = synth.tiny()
    w = synth.make_weights(wl.dims, wl.seed)
    out = _run(wl, w)
    with open(os.path.join(HERE, "tiny_actions.txt"), "w") as f:
        f.write("# oracle actions of the 2-layer fp32 tiny case, seed 0, 2 Euler steps; [16 x 8]\n")
        np.savetxt(f, out.reshape(-1, wl.dims.action_dim), fmt="%.17g")


def pad2048():
    w = synth.make_weights(synth.PI05, 0)
    rows, lens = [], []
    for seed in SEEDS:
        t = time.time()
        wl = synth.pi05_padded(seed, padded=False)
        rows.append(_run(wl, w).reshape(-1, synth.PI05.action_dim))
        lens.append(wl.n_valid[0])
        print(f"pad2048 seed {seed}: {wl.n_valid[0]} valid rows, {time.time() - t:.1f} s", flush=True)
    header = ("oracle actions, Pi0.5-shaped expert (weights seed 0), one request of the 2048-padded "
              f"workload per seed {list(SEEDS)} (valid rows {lens}), 10 Euler steps; "
              "[seeds * 50, 32], seed-major")
    np.savetxt(os.path.join(HERE, "pi05_pad2048_actions.txt.gz"), np.concatenate(rows), fmt="%.9g",
               header=header)


def batched():
    w = synth.make_weights(synth.PI05, 0)
    rows = []
    for seed in SEEDS:
        t = time.time()
        wl = synth.pi05_batched(seed)
        rows.append(_run(wl, w).reshape(-1, synth.PI05.action_dim))
        print(f"batched seed {seed}: lengths {wl.n_valid}, {time.time() - t:.1f} s", flush=True)
    header = ("oracle actions, Pi0.5-shaped expert (weights seed 0), 16 requests of 600..2048 valid "
              f"prefix rows per seed {list(SEEDS)}, 10 Euler steps; [seeds * 16 * 50, 32], "
              "seed-major then request-major")
    np.savetxt(os.path.join(HERE, "pi05_b16_ragged_actions.txt.gz"), np.concatenate(rows), fmt="%.9g",
               header=header)


def main(argv):
    jobs = {"tiny": tiny, "pad2048": pad2048, "batched": batched}
    for name in (argv or list(jobs)):
        jobs[name]()


if __name__ == "__main__":
    main(sys.argv[1:])
