"""Write tests/golden/small_case.json.  Calls only oracle/ (and the seeded
input generators in q8_synth); nothing here comes from the CUDA library.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import q8_synth  # noqa: E402


def main():
    N, K, M, seed_w, seed_x = 9, 96, 2, 101, 202
    W = oracle.quantize(q8_synth.weights(N, K, seed_w).numpy())
    A = oracle.quantize(q8_synth.activations(M, K, seed_x).numpy())
    isum = oracle.block_dots(W, A, K)
    y, S = oracle.gemm(W, A, K)
    out = {
        "what": "small seeded case: W 9x96 ~N(0,0.02), x 2x96 ~N(0,1), numpy PCG64",
        "N": N, "K": K, "M": M, "seed_w": seed_w, "seed_x": seed_x,
        "W_blocks_hex": W.tobytes().hex(),
        "A_blocks_hex": A.tobytes().hex(),
        "isum": isum.ravel().tolist(),
        "y": [float(v) for v in y.ravel()],
        "S": [float(v) for v in S.ravel()],
    }
    with open(os.path.join(HERE, "small_case.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
