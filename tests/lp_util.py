"""Helpers shared by the tests: move synthetic inputs to the GPU and compare with the oracle."""
import numpy as np

import synth


def part_of(p):
    import lm_head_linear_tcgen05_gb300 as lp
    return lp.VocabPartition(p.vocab_real, p.vocab_padded, tuple(p.ranges))


def dev_bf16(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def dev_i32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def dev_f32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_inputs(inp: synth.ForwardInputs, device="cuda"):
    X = dev_bf16(inp.X, device)
    W = [dev_bf16(w, device) if w.shape[0] > 0 else None for w in inp.W]
    b = None if inp.bias is None else [dev_bf16(x, device) if x.shape[0] > 0 else None for x in inp.bias]
    return X, W, b, dev_i32(inp.y, device)


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    d = np.abs(np.where(both_inf, 0.0, a) - np.where(both_inf, 0.0, b))
    return float(np.max(d)) if d.size else 0.0


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


# tolerances of the GPU path against the fp64 oracle
TOL_LOGP = 2e-3
TOL_LSE = 2e-3
TOL_ENT = 5e-3
TOL_GRAD_REL = 1e-2
