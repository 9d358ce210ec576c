"""Helpers for the GPU parity tests: seeded inputs, oracle comparison."""
import numpy as np
import torch

from long_context_sequence_seq_gb300 import inputs

TOL = {"bf16": 2e-2, "fp32": 1e-4}
LSE_TOL = {"bf16": 1e-3, "fp32": 1e-4}


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def seq_inputs(S, Hq, Hkv, D, dtype, B=1, seed_offset=0, device="cuda"):
    """Seeded N(0,1) Q, K, V, dO in sequence layout, drawn on the host."""
    shp_q, shp_k = (B, S, Hq, D), (B, S, Hkv, D)
    t = [inputs.host_tensor(shp_q, inputs.SEED_Q + seed_offset, dtype),
         inputs.host_tensor(shp_k, inputs.SEED_K + seed_offset, dtype),
         inputs.host_tensor(shp_k, inputs.SEED_V + seed_offset, dtype),
         inputs.host_tensor(shp_q, inputs.SEED_DO + seed_offset, dtype)]
    return [x.to(device) for x in t]


def max_err(got, want):
    return float(np.max(np.abs(got - want))) if got.size else 0.0


def to_head_np(x_seq):
    """[B,S,H,D] numpy -> [B,H,S,D] (a view used only to feed the oracle)."""
    return np.ascontiguousarray(np.transpose(x_seq, (0, 2, 1, 3)))
