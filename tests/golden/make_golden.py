"""Write tests/golden/tiny_recurrence.json: a fixed small input (numpy seed 20) and
the fp64 oracle's output on it.  Calls only oracle/; rerun after a deliberate change
to the oracle's arithmetic and say in the commit which passage justifies it."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(20)
    B, T, H, K, V = 1, 6, 2, 4, 3
    f32 = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, k, v = f32(B, T, H, K), f32(B, T, H, K), f32(B, T, H, V)
    g = (-rng.random((B, T, H, K)) * 2).astype(np.float32)
    beta = rng.random((B, T, H)).astype(np.float32)
    s0 = rng.standard_normal((B, H, K, V)) * 0.1
    scale = 0.5
    o, s = oracle.recurrent(q, k, v, g, beta, s0, scale=scale)
    out = {
        "description": "Regression values of the fp64 oracle (kernel L2 norm on, eps 1e-6) written by make_golden.py",
        "inputs": {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "g": g.tolist(), "beta": beta.tolist(),
                   "initial_state": s0.tolist(), "scale": scale},
        "expected": {"o": o.tolist(), "final_state": s.tolist()},
    }
    with open(os.path.join(HERE, "tiny_recurrence.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
