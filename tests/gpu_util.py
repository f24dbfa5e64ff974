"""Helpers shared by the GPU tests: moving seeded numpy inputs to the device
and comparing library outputs with the oracle at the stated tolerances.

Tolerances (fixed before any kernel was run): per-token nll within 4e-3
absolute, summed bits per byte within 1e-5 relative, dh and dW within 1e-2
relative Frobenius error, int4 dequantisation bit-exact.
"""
import numpy as np
import torch

NLL_ATOL = 4e-3
BPB_RTOL = 1e-5
GRAD_RTOL = 1e-2


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_inputs(inp: dict) -> dict:
    out = dict(h=bf16_dev(inp["h"]), W=bf16_dev(inp["W"]),
               tgt=torch.from_numpy(inp["tgt"]).cuda(),
               nbytes=torch.from_numpy(inp["nbytes"]).cuda(),
               mask=None if inp["mask"] is None else torch.from_numpy(inp["mask"]).cuda())
    if "Wq" in inp:
        out["Wq"] = torch.from_numpy(inp["Wq"]).cuda()
        out["scales"] = torch.from_numpy(inp["scales"].view(np.int16)).cuda()
    return out


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
