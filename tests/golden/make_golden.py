"""Write the oracle's output for the tiny 256x256, 4-bit, seed-0 layer.

Calls only oracle/ and the seeded input module. Run from the repository root:
    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

K = N = 256
BITS = 4
t = synth.codes(0, K, N, BITS)
y = oracle.linear(t, K, N, BITS, synth.suh(0, K).astype(np.float64), synth.svh(0, N).astype(np.float64),
                  synth.as_f64(synth.activations(0, 1, K), "f16"))
out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_k256_n256_b4_seed0.txt")
np.savetxt(out, y[0], fmt="%.17g",
           header="oracle y of K=N=256, bits=4, rows=1, seed 0 (synth recipe); written by make_golden.py")
print(out)
