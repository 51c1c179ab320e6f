"""Writes oracle_small_case.txt: the oracle's outputs for one small, fully specified case, so
that any later change to the oracle's arithmetic shows up as a diff here (a change must name
the passage or reading that justifies it). Calls only oracle/ on inputs defined below."""

import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle.attention import ACC_FP32, GRAN_PER_THREAD, sage_attention  # noqa: E402


def case_inputs():
    """B=1, H=1, Nq=Nk=6, d=4: small integer patterns scaled by 1/8 (exact in fp32)."""
    i = np.arange(6)[:, None]
    c = np.arange(4)[None, :]
    q = (((3 * i + 5 * c) % 7) - 3) / 8.0
    k = (((2 * i + 3 * c) % 5) - 2) / 8.0 + np.array([0.5, -0.25, 0.0, 1.0])[None, :]
    v = (((i + 2 * c) % 6) - 2.5) / 4.0
    return (q[None, None].astype(np.float32), k[None, None].astype(np.float32),
            v[None, None].astype(np.float32))


def compute():
    q, k, v = case_inputs()
    out = {}
    for causal in (False, True):
        r = sage_attention(q, k, v, is_causal=causal, gran=GRAN_PER_THREAD, accum=ACC_FP32,
                           smooth_k=True, smooth_v=True)
        out[causal] = (r["o"][0, 0], r["lse"][0, 0])
    return out


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.txt")
    with open(path, "w") as f:
        f.write("# oracle outputs for make_oracle_case.case_inputs(): per_thread INT8, fp32\n")
        f.write("# accumulation, smooth_k and smooth_v on; rows: 'o <causal> <row> 4 values',\n")
        f.write("# 'lse <causal> <row> value'; float64 values as hex floats.\n")
        for causal, (o, lse) in compute().items():
            for r in range(o.shape[0]):
                f.write(f"o {int(causal)} {r} " + " ".join(float(x).hex() for x in o[r]) + "\n")
            for r in range(lse.shape[0]):
                f.write(f"lse {int(causal)} {r} {float(lse[r]).hex()}\n")


if __name__ == "__main__":
    main()
