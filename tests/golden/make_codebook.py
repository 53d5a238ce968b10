"""Write ``codebook_seed0.json``: the Lloyd-Max Gaussian codebooks fitted by the oracle.

The table is the ``cb2[4] | cb3[8] | cb4[16]`` header table of the Needle .cact page,
§一 (Lloyd-Max on 400,000 Gaussian samples, 200 iterations).  The samples are drawn by
``gemm_cq_gemv_gb300.synth.gaussian_samples(seed=0)``; every number in the output comes
from ``oracle.lloyd_max_gaussian_fit``.  Parity tests feed this table to both the CUDA
path and the oracle, so bit-exact encode parity never depends on a fit.

Run from the repository root:  python tests/golden/make_codebook.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from gemm_cq_gemv_gb300.synth import gaussian_samples, LLOYD_MAX_SAMPLES  # noqa: E402
from oracle import lloyd_max_gaussian_fit  # noqa: E402


def build():
    s = gaussian_samples(LLOYD_MAX_SAMPLES, seed=0)
    out = {"samples": LLOYD_MAX_SAMPLES, "seed": 0, "iterations": 200}
    for b, L in ((2, 4), (3, 8), (4, 16)):
        lv = lloyd_max_gaussian_fit(s, L, 200)
        out[f"cb{b}"] = [float(v) for v in lv]
        out[f"cb{b}_f32_hex"] = [format(int(v), "08x") for v in lv.view("uint32")]
    return out


if __name__ == "__main__":
    data = build()
    with open(os.path.join(HERE, "codebook_seed0.json"), "w") as f:
        json.dump(data, f, indent=1)
    print("wrote codebook_seed0.json")
