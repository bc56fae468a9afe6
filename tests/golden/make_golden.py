"""Write tests/golden/oracle_regression.json from the oracle alone.

The fixture freezes the oracle's output on a small, platform-independent
input (bf16 bit patterns from a 64-bit LCG), so the aarch64 GPU host and the
x86_64 build host can be checked to compute the same bits.  It is a
regression fixture for the oracle, not a pin against the method: the pins
are in tests/test_oracle.py.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")


def lcg_bf16(n, seed):
    """n bf16 bit patterns with exponent in [2^-8, 2^1] and random sign."""
    out = np.empty(n, np.uint16)
    s = seed & 0xFFFFFFFFFFFFFFFF
    for i in range(n):
        s = (s * 6364136223846793005 + 1442695040888963407) & 0xFFFFFFFFFFFFFFFF
        r = s >> 33
        sign = (r >> 20) & 1
        exp = 119 + (r >> 8) % 10  # biased exponents 119..128
        mant = r & 0x7F
        out[i] = (sign << 15) | (exp << 7) | mant
    return out


def inputs():
    K, N, M = 16, 6, 5
    X = lcg_bf16(K * N, 1).reshape(K, N)
    D = lcg_bf16(K * M, 2).reshape(K, M)
    W = (oracle.decode(lcg_bf16(N * M, 3)) * 0.01).astype(np.float32).reshape(N, M)
    m = (oracle.decode(lcg_bf16(N * M, 4)) * 1e-3).astype(np.float32).reshape(N, M)
    v = np.abs(oracle.decode(lcg_bf16(N * M, 5)) * 1e-4).astype(np.float32).reshape(N, M)
    return K, N, M, X, D, W, m, v


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def compute():
    K, N, M, X, D, W, m, v = inputs()
    G = oracle.wgrad(X, D)
    a = oracle.adamw(G, W, m, v, step=4, **HP)
    b = oracle.adamw(G, W, oracle.round_bf16(m), oracle.round_bf16(v), step=4, **HP)
    s = oracle.sgdm(G, W, m, lr=1e-2, momentum=0.9, wd=0.0)
    off = np.array([0, 5, 5, 16])
    Wg = np.stack([W, W * 2, W * 3]).astype(np.float32)
    mg = np.stack([m, m, m])
    vg = np.stack([v, v, v])
    g = oracle.grouped_adamw(X, D, off, Wg, mg, vg, step=2, **HP)
    return {
        "G_f64_hex": [float(x).hex() for x in G.ravel()],
        "adamw_f32": {"W": a["W"].view(np.uint32).ravel().tolist(),
                      "m": a["m"].view(np.uint32).ravel().tolist(),
                      "v": a["v"].view(np.uint32).ravel().tolist()},
        "adamw_bf16": {"W": b["W"].view(np.uint32).ravel().tolist(),
                       "m": b["m"].ravel().tolist(), "v": b["v"].ravel().tolist()},
        "sgdm_f32": {"W": s["W"].view(np.uint32).ravel().tolist(),
                     "buf": s["buf"].view(np.uint32).ravel().tolist()},
        "grouped_f32": {"W": g["W"].view(np.uint32).ravel().tolist(),
                        "m": g["m"].view(np.uint32).ravel().tolist(),
                        "v": g["v"].view(np.uint32).ravel().tolist()},
    }


if __name__ == "__main__":
    doc = {
        "what": "oracle regression fixture: K=16, N=6, M=5 bf16 LCG inputs; AdamW step 4 "
                "(lr 1e-3, betas 0.9/0.999, eps 1e-8, wd 0.01) in fp32 and bf16 state; "
                "SGD momentum 0.9 lr 1e-2; grouped with token offsets [0,5,5,16]",
        "written_by": "tests/golden/make_golden.py (calls only oracle/)",
        "data": compute(),
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", OUT)
