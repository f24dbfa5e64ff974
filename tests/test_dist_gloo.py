"""Multi-rank host logic on CPU: two gloo ranks each score a contiguous row
shard (with the CPU oracle standing in for a GPU's forward), add their input
positions' embedding gradients into the same table gradient, then combine
the bits-per-byte sums and dW; the result equals the single-process answer
(head dW plus every position's embedding gradient).  Also: a loop whose stop
condition differs per rank runs the same number of collective steps on every
rank when the ranks decide with dist.any_rank (the benchmark's warm-up)."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_path):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    import synth_inputs as si
    from lm_head_softcapped_lmhead_b300 import dist as ld

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = si.make_inputs(2, N=101, V=64, d=64, w_scale=10.0)
    a, b = ld.row_shard(inp["N"], rank, world)
    nll, lse = oracle.fwd(inp["h"][a:b], inp["W"], inp["tgt"][a:b], 30.0)
    _, sn, sb, n = oracle.bpb(nll, inp["nbytes"][a:b])
    tot = ld.allreduce_bpb((sn, sb, n))
    _, dW = oracle.bwd(inp["h"][a:b], inp["W"], inp["tgt"][a:b], 30.0, lse, 1.0 / inp["N"], want_dh=False)
    # the rank's input positions' embedding gradients join the same table gradient before the exchange
    e = si.make_embed_inputs(N=101, V=64, d=64, seed=77)
    dW = dW + oracle.embed_bwd(e["ids"][a:b], e["g"][a:b], 64)
    dWt = torch.from_numpy(dW)
    ld.allreduce_dW(dWt)
    # the accumulator exchange the benchmark uses (24 bytes per rank, combined in rank order)
    acc = torch.tensor([sn, 0.0, 0.0], dtype=torch.float64)
    acc.view(torch.int64)[1] = sb
    acc.view(torch.int64)[2] = n
    tot2 = ld.combine_bpb_acc(ld.allgather_bpb_acc(acc))
    # A loop whose stop condition differs per rank (the benchmark's timed
    # warm-up) runs the same number of steps everywhere when the ranks decide
    # together: here rank 1 would stop after 3 steps and rank 0 after 11.
    steps = 0
    while ld.any_rank(steps < (11 if rank == 0 else 3)):
        dist.all_reduce(torch.ones(1))  # a step's collective
        steps += 1
    agree = [ld.any_rank(rank == 0), ld.any_rank(False)]
    counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(counts, torch.tensor([steps]))
    if rank == 0:
        np.savez(out_path, sn=tot[0], sb=tot[1], n=tot[2], dW=dWt.numpy(), sn2=tot2[0], sb2=tot2[1], n2=tot2[2],
                 steps=np.array([int(c) for c in counts]), agree=np.array(agree))
    dist.barrier()
    dist.destroy_process_group()


def test_row_shard_partition():
    from lm_head_softcapped_lmhead_b300.dist import row_shard
    for N in (1, 7, 100, 65536):
        for world in (1, 2, 3, 8):
            spans = [row_shard(N, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_single_process(tmp_path, oracle_mod):
    import synth_inputs as si
    out = str(tmp_path / "r0.npz")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    got = np.load(out)
    inp = si.make_inputs(2, N=101, V=64, d=64, w_scale=10.0)
    nll, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    b, sn, sb, n = oracle_mod.bpb(nll, inp["nbytes"])
    assert int(got["sb"]) == sb and int(got["n"]) == n
    assert float(got["sn"]) == pytest.approx(sn, rel=1e-13)
    assert (float(got["sn2"]), int(got["sb2"]), int(got["n2"])) == (float(got["sn"]), int(got["sb"]), int(got["n"]))
    _, dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, lse, 1.0 / inp["N"], want_dh=False)
    e = si.make_embed_inputs(N=101, V=64, d=64, seed=77)
    dW = dW + oracle_mod.embed_bwd(e["ids"], e["g"], 64)
    assert np.allclose(got["dW"], dW, rtol=0, atol=1e-14)
    assert list(got["steps"]) == [11, 11]
    assert list(got["agree"]) == [True, False]
