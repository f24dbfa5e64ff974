"""Writes the stored oracle outputs the tests compare against.  Every value
comes from the fp64 CPU oracle (``oracle/``) on seeded synthetic inputs
(``synth_inputs``); no CUDA code is imported.  Re-run after a deliberate,
justified change of the oracle's arithmetic:

    python tests/golden/make_golden.py            # oracle_small.json (seconds)
    python tests/golden/make_golden.py --full     # also full_size.json (~2 min on 8 cores)

oracle_small.json: small cases (per-row nll and bpb).
full_size.json: the workloads at full size, for the GPU parity tests --
  * the forward + backward batch (N = 16384) and the training micro-batch
    (N = 65536), V = 8192, softcap 30, mean loss: the whole batch's sums of
    nll and bytes and its bpb, and dW (grad_scale 1/N) on 8 vocabulary rows:
    the four most frequent Zipf targets (ids 0-3), two mid-frequency ids and
    two rare ones;
  * the int4 head (N = 65536): the batch's sums and bpb with the head
    dequantised by the oracle;
  * the sliding-window evaluation stream: 8 chunks of 32 windows (65,536 rows,
    2,048 scored each), per chunk the sums of nll and bytes over the scored
    rows, and the bpb of the 8 chunks together.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402

CASES = [
    dict(cfg=1, N=16, V=64, d=64, w_scale=1.0, softcap=30.0),
    dict(cfg=2, N=16, V=96, d=128, w_scale=100.0, softcap=30.0),
    dict(cfg=2, N=8, V=40, d=64, w_scale=50.0, softcap=2.0),
]

SOFTCAP = 30.0
VROWS = [0, 1, 2, 3, 100, 1000, 5000, 8191]
STREAM_CHUNKS = 8


def small():
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


def batch_entry(cfg):
    inp = si.make_inputs(cfg)
    N = inp["N"]
    W = inp["W"] if cfg != 5 else oracle.dequant_int4(inp["Wq"], inp["scales"], inp["d"], si.INT4_GROUP)
    nll, lse = oracle.fwd(inp["h"], W, inp["tgt"], SOFTCAP)
    b, sn, sb, n = oracle.bpb(nll, inp["nbytes"])
    e = dict(N=N, V=inp["V"], d=inp["d"], seed=inp["seed"], softcap=SOFTCAP,
             sum_nll=sn, sum_bytes=sb, n_scored=n, bpb=b)
    if cfg != 5:
        w = 1.0 / N
        rows = oracle.dW_rows(inp["h"], W, inp["tgt"], SOFTCAP, lse, w, np.array(VROWS))
        counts = np.bincount(inp["tgt"], minlength=inp["V"])
        e.update(grad_scale=w, vrows=VROWS, vrow_target_counts=[int(counts[v]) for v in VROWS],
                 dW_rows=[[float(f"{x:.10e}") for x in r] for r in rows])
    return e


def stream_entry():
    chunks = []
    tot_nll, tot_b = 0.0, 0
    for k in range(STREAM_CHUNKS):
        inp = si.make_stream_chunk(k)
        sel = np.nonzero(inp["mask"])[0]
        nll, _ = oracle.fwd(inp["h"], inp["W"], inp["tgt"], SOFTCAP, rows=sel)
        b, sn, sb, n = oracle.bpb(nll, inp["nbytes"][sel])
        chunks.append(dict(k=k, seed=inp["seed"], rows=int(inp["N"]), sum_nll=sn, sum_bytes=sb, n_scored=n))
        tot_nll += sn
        tot_b += sb
    return dict(windows_per_chunk=si.STREAM_CHUNK_WINDOWS, softcap=SOFTCAP, chunks=chunks,
                bpb=tot_nll / (np.log(2.0) * tot_b))


def full():
    out = {"note": "fp64 CPU oracle outputs at full workload sizes (synth_inputs seeds); "
                   "written by tests/golden/make_golden.py --full",
           "cfg2": batch_entry(2), "cfg3": batch_entry(3), "cfg5": batch_entry(5),
           "cfg4_stream": stream_entry()}
    with open(os.path.join(HERE, "full_size.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    small()
    if "--full" in sys.argv:
        full()
