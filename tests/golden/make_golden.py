"""Writes oracle_small.json: small seeded cases run through the CPU oracle
only (no CUDA code is imported).  Re-run after a deliberate, justified change
of the oracle's arithmetic:  python tests/golden/make_golden.py"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402

CASES = [
    dict(cfg=1, N=16, V=64, d=64, w_scale=1.0, softcap=30.0),
    dict(cfg=2, N=16, V=96, d=128, w_scale=100.0, softcap=30.0),
    dict(cfg=2, N=8, V=40, d=64, w_scale=50.0, softcap=2.0),
]


def main():
    out = {"note": "fp64 CPU oracle outputs for seeded synthetic inputs "
                   "(synth_inputs.make_inputs); written by make_golden.py",
           "cases": []}
    for c in CASES:
        inp = si.make_inputs(c["cfg"], N=c["N"], V=c["V"], d=c["d"], w_scale=c["w_scale"])
        nll, lse = oracle.fwd(inp["h"], inp["W"], inp["tgt"], c["softcap"])
        b, *_ = oracle.bpb(nll, inp["nbytes"])
        out["cases"].append(dict(c, nll=[float(x) for x in nll], bpb=b))
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
