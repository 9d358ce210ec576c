"""Helpers for the GPU parity tests: seeded inputs, oracle comparison."""
import math

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


def bf16_rounding_bound(q, k, v, do, cu_seqlens=None, causal=True):
    """Element-wise worst-case error the bf16 tensor-core path can add on top
    of fp32 accumulation, for one batch entry: q, do [H_q, S, D], k, v
    [H_kv, S, D] in fp64 (the bf16 inputs, exactly).

    The kernels feed the second-stage MMAs bf16 operands, as the bf16-input /
    fp32-accumulate contract implies: P = bf16(exp(s - LSE)) for O and dV, and
    dS = bf16(P (dP - D)) for dQ and dK, with D_i computed from the
    bf16-rounded O.  With u = 2^-8 (the unit roundoff of bf16's 8-bit
    significand: round-to-nearest errs by at most u relative):
      b_i     = u sum_j P_ij |v_j| + u |O_i|   bounds the error of O_i (also stored as bf16)
      |dV_j| <= u sum_i P_ij |dO_i|
      e_ij    = u |dS_ij| + P_ij sum_d |dO_id| b_id       (D_i is formed from that O)
      |dQ_i| <= scale sum_j e_ij |k_j|,  |dK_j| <= scale sum_i e_ij |q_i|
    element by element (dK/dV summed over the q heads of a kv head).  These
    bounds assume every rounding error points the same way, so the measured
    error sits well inside them; they scale with the gradients' magnitudes,
    which the fixed 2e-2 of the N(0,1) workloads does not.  Returns bounds for
    (O, dQ, dK, dV) shaped like those tensors."""
    from oracle import key_ranges      # the mask only: row i sees keys [lo_i, hi_i)
    Hq, S, D = q.shape
    G = Hq // k.shape[0]
    sc = 1.0 / math.sqrt(D)
    u = 2.0 ** -8
    lo, hi = key_ranges(S, cu_seqlens, causal)
    j = np.arange(S)
    allowed = (j[None, :] >= lo[:, None]) & (j[None, :] < hi[:, None])
    b_o, b_q = np.zeros(q.shape), np.zeros(q.shape)
    b_k, b_v = np.zeros(k.shape), np.zeros(k.shape)
    for h in range(Hq):
        g = h // G
        s = np.where(allowed, sc * (q[h] @ k[g].T), -np.inf)
        e = np.exp(s - s.max(axis=1)[:, None])
        p = e / e.sum(axis=1)[:, None]
        o = p @ v[g]
        dp = do[h] @ v[g].T
        ds = p * (dp - np.sum(p * dp, axis=1)[:, None])
        b_o[h] = u * (p @ np.abs(v[g])) + u * np.abs(o)
        err_s = u * np.abs(ds) + p * np.sum(np.abs(do[h]) * b_o[h], axis=1)[:, None]
        b_q[h] = sc * (err_s @ np.abs(k[g]))
        b_k[g] += sc * (err_s.T @ np.abs(q[h]))
        b_v[g] += u * (p.T @ np.abs(do[h]))
    return b_o, b_q, b_k, b_v
