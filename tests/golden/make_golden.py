"""Write the oracle regression fixtures in this folder.

Calls only the float64 oracle (``oracle/``) on small seeded inputs drawn by
``chunkwise_gated_delta_gdr_gb300.inputs`` and stores the outputs as text, so
that a later change to the oracle's arithmetic shows up as a diff. Run from the
repository root: ``python tests/golden/make_golden.py``.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from chunkwise_gated_delta_gdr_gb300 import inputs as gin  # noqa: E402

CASES = {
    # name: (workload, overrides)
    "oracle_gdn_small": ("gdn_t4096_h12", dict(T=21, H=2, HV=2, K=8, V=6, C=8)),
    "oracle_kda_gqa_small": ("kda_gqa_t8192", dict(B=1, T=13, H=1, HV=2, K=8, V=4, C=4)),
    "oracle_long_state_small": ("gdn_long_t65000", dict(T=11, H=1, HV=1, K=6, V=5, C=4)),
}


def compute(name):
    wname, ov = CASES[name]
    w = gin.shrink(gin.WORKLOADS[wname], **ov)
    x = gin.make_inputs(w)
    o, S = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale)
    return w, o, S


def write(name):
    w, o, S = compute(name)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), name + ".txt")
    with open(path, "w") as f:
        f.write(f"# oracle regression fixture: workload {w.name} shrunk to "
                f"B={w.B} T={w.T} H={w.H} HV={w.HV} K={w.K} V={w.V}\n")
        f.write("# written by tests/golden/make_golden.py from oracle.recurrent (float64)\n")
        f.write(f"o_shape {' '.join(map(str, o.shape))}\n")
        f.write("o " + " ".join(repr(float(x)) for x in o.ravel()) + "\n")
        f.write(f"S_shape {' '.join(map(str, S.shape))}\n")
        f.write("S " + " ".join(repr(float(x)) for x in S.ravel()) + "\n")


def read(name):
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), name + ".txt")
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = rest
    o = np.array([float(x) for x in vals["o"]]).reshape([int(x) for x in vals["o_shape"]])
    S = np.array([float(x) for x in vals["S"]]).reshape([int(x) for x in vals["S_shape"]])
    return o, S


if __name__ == "__main__":
    for n in CASES:
        write(n)
        print("wrote", n)
