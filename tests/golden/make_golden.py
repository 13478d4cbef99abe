"""Writes tiny_oracle_summary.json: a regression record of the fp64 oracle on the tiny workload.

The pages print no worked numeric example, so nothing here comes from them; this record only
guards the oracle against unintended changes.  It calls nothing but ``oracle`` and ``synth``.
Run from the repository root:  python -m tests.golden.make_golden
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def summarise():
    cfg = synth.CONFIGS["tiny"]
    L = oracle.Layer(synth.make_inputs(cfg, seed=0), cfg)
    y, _ = L.forward()
    g = L.backward()
    D = L.dispatch()
    norms = {"y": float(np.sqrt(np.sum(y * y)))}
    for key in ("dx", "dW_r", "dW_gate", "dW_up", "dW_down", "dgates"):
        norms[key] = float(np.sqrt(np.sum(g[key] * g[key])))
    norms["gates"] = float(np.sqrt(np.sum(L.routing().gates ** 2)))
    # the e4m3 forward and backward, and the MX conversion, on the same workload
    from oracle import fp8
    y8 = fp8.layer_forward_fp8(L)
    g8 = fp8.layer_backward_fp8(L)
    norms["fp8_y"] = float(np.sqrt(np.sum(y8 * y8)))
    for key in ("dx", "dW_gate", "dW_up", "dW_down", "dgates"):
        norms["fp8_" + key] = float(np.sqrt(np.sum(g8[key] * g8[key])))
    xq, xs = fp8.quantize_rows_e4m3(L.x[:2].astype(np.float32))
    mq, me = fp8.mx_quantize_e4m3(L.x[:2].astype(np.float32))
    return {"counts": [int(c) for c in D.counts],
            "idx_head": L.routing().idx[:8].tolist(),
            "fp8_x_codes_head": xq[:, :16].tolist(),
            "fp8_x_scales_head": [float(v) for v in xs],
            "mx_x_codes_head": mq[:, :16].tolist(),
            "mx_x_exps": me.tolist(),
            "norms": norms}


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_summary.json")
    with open(out, "w") as fh:
        json.dump({"about": __doc__.strip().splitlines()[0], **summarise()}, fh, indent=1)
    print("wrote", out)
