"""Write the oracle regression fixtures in this folder.

The pages (deepseek_v4.py of sglang, and prefill_sp.py / test_prefill_sp_gpu.py
of the recipes repo) print no worked numeric example of the hyper-connection
work, so no fixture here holds a value from the pages.  What this script
stores is the oracle's own output on the first rows of the 128-row seed-0
workload, so that any later change to the oracle's arithmetic shows up as a
failing test and has to be justified.  It calls only ``oracle`` (and ``synth``
for the seeded inputs) -- never the CUDA path.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

ROWS = 8


def digest(a) -> str:
    return hashlib.sha256(a.tobytes()).hexdigest()


def main():
    R = synth.residual(0, ROWS)
    W = synth.weights(0)
    y = synth.sublayer_out(0, ROWS)
    o = oracle.pre(R, W.fn, W.scale, W.base, W.norm_w)
    post32 = o["post"].astype("float32")
    comb32 = o["comb"].astype("float32")
    r_out = oracle.post(R, y, post32, comb32)
    q, sc = oracle.mxfp8_quantize(o["x_norm"])
    fixture = {
        "what": "oracle outputs on rows 0..7 of the M=128 seed-0 workload (regression only)",
        "inputs": {"seed": 0, "rows": ROWS, "rms_eps": 1e-6, "hc_pre_eps": 1e-6,
                   "hc_sinkhorn_eps": 1e-6, "norm_eps": 1e-6, "post_mult": 2.0, "iters": 20,
                   "R_sha256": digest(R), "y_sha256": digest(y)},
        "mix": o["mix"].tolist(),
        "pre": o["pre"].tolist(),
        "post": o["post"].tolist(),
        "comb": o["comb"].tolist(),
        "x_norm_sha256": digest(o["x_norm"]),
        "x_norm_row0_first8": [int(v) for v in o["x_norm"][0, :8]],
        "r_out_sha256": digest(r_out),
        "r_out_row0_stream1_first8": [int(v) for v in r_out[0, 1, :8]],
        "x_norm_mxfp8_codes_sha256": digest(q),
        "x_norm_mxfp8_scales_sha256": digest(sc),
        "x_norm_mxfp8_scales_row0": [int(v) for v in sc[0]],
        "x_norm_mxfp8_scales_128x4_sha256": digest(oracle.swizzle_128x4(sc)),
    }
    with open(os.path.join(HERE, "oracle_m128_seed0_rows0-7.json"), "w") as f:
        json.dump(fixture, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
