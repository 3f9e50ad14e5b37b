"""Write the stored oracle outputs under tests/golden/.

Calls only the oracle and the seeded input generator; no value here comes from
the CUDA library.  Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from flow_matching_action_gb300 import synth  # noqa: E402
from oracle import ae_oracle  # noqa: E402


def main():
    wl = synth.tiny()
    w = synth.make_weights(wl.dims, wl.seed)
    out = ae_oracle.sample(wl.dims, w, wl.prefix_k, wl.prefix_v, wl.cu_lens, wl.mask, wl.noise, wl.n_steps)
    with open(os.path.join(HERE, "tiny_actions.txt"), "w") as f:
        f.write("# oracle actions of the 2-layer fp32 tiny case, seed 0, 2 Euler steps; [16 x 8]\n")
        np.savetxt(f, out.reshape(-1, wl.dims.action_dim), fmt="%.17g")


if __name__ == "__main__":
    main()
