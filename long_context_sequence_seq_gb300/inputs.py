"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds workload shapes and random-number recipes only: no attention
or re-layout arithmetic lives here, so the oracle and the CUDA path can both use
it without sharing any of the method's code.

Workloads (Ulysses sequence parallelism, "How it works" steps 1-5 of
"Ulysses Sequence Parallelism: Training with Million-Token Contexts"):

  tiny_mha_fp32      S=256,   H_q=H_kv=8,  D=64,  P=2, fp32, head_chunk=4
  qwen3_4b_8k        S=8192,  H_q=32, H_kv=8, D=128, P=4, bf16, head_chunk=8
  qwen3_4b_64k       S=65536, same layer, head_chunk=8 (headline point)
  llama31_8b_packed  S=131072 packed documents, log-uniform lengths in
                     [512, 32768] (last one truncated), P=8, head_chunk=4
  million_token      S=1048576, P=8, head_chunk=4

Inputs are N(0,1).  fp32 values are drawn first and cast to bf16 with
round-to-nearest-even (torch's ``.to(torch.bfloat16)``).  Seeds: Q=0, K=1,
V=2, dO=3, document lengths=4.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_DOCS = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int
    H_q: int
    H_kv: int
    D: int
    P: int
    head_chunk: int
    dtype: str  # "bf16" or "fp32"
    packed: bool = False
    B: int = 1
    causal: bool = True
    hidden: int = 0   # model width for the projection GEMMs (0: none given)

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv


WORKLOADS = {
    "tiny_mha_fp32": Workload("tiny_mha_fp32", 256, 8, 8, 64, 2, 4, "fp32"),
    "qwen3_4b_8k": Workload("qwen3_4b_8k", 8192, 32, 8, 128, 4, 8, "bf16", hidden=2560),
    "qwen3_4b_64k": Workload("qwen3_4b_64k", 65536, 32, 8, 128, 4, 8, "bf16", hidden=2560),
    "llama31_8b_packed": Workload("llama31_8b_packed", 131072, 32, 8, 128, 8, 4,
                                  "bf16", packed=True),
    "million_token": Workload("million_token", 1048576, 32, 8, 128, 8, 4, "bf16"),
}


def doc_lengths(S: int, seed: int = SEED_DOCS, lo: int = 512, hi: int = 32768):
    """Document lengths floor(exp(U[ln lo, ln hi))) drawn until they cover S.

    The last document is truncated so the lengths sum to exactly S (it may end
    up shorter than ``lo``).  Packing several documents into one sequence is
    what the TRL SFTTrainer "packing" option does.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = []
    total = 0
    while total < S:
        L = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        L = max(1, min(L, S - total))
        lengths.append(L)
        total += L
    return lengths


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def workload_cu_seqlens(w: Workload):
    """int32 cu_seqlens for a packed workload, else None (one causal document)."""
    if not w.packed:
        return None
    return cu_seqlens_from_lengths(doc_lengths(w.S))


def host_normal(shape, seed: int) -> np.ndarray:
    """fp32 N(0,1) from numpy PCG64 (used for small shapes)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal(size=shape, dtype=np.float32)


def host_tensor(shape, seed: int, dtype: str):
    """A torch CPU tensor of N(0,1) values in the workload dtype.

    bf16 values are the round-to-nearest-even cast of the fp32 draw.
    """
    import torch
    x = torch.from_numpy(host_normal(shape, seed))
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "fp32":
        return x
    raise ValueError(dtype)


def device_tensor(shape, seed: int, dtype: str, device="cuda"):
    """N(0,1) drawn on the device with a seeded torch generator (large shapes)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.empty(shape, dtype=torch.float32, device=device)
    # draw in slabs to bound the fp32 temporary
    flat = x.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        flat[i:i + step].normal_(generator=g)
    if dtype == "bf16":
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        fo = out.view(-1)
        for i in range(0, flat.numel(), step):
            fo[i:i + step].copy_(flat[i:i + step])
        del x
        return out
    return x


def seq_shapes(w: Workload):
    """Sequence-layout shapes [B, S, H, D] of Q, K/V and dO (one per rank chunk)."""
    return ((w.B, w.S, w.H_q, w.D), (w.B, w.S, w.H_kv, w.D), (w.B, w.S, w.H_q, w.D))


def make_seq_inputs(w: Workload, device=None, small_on_host: bool = True):
    """Q, K, V, dO in sequence layout [B, S, H, D].

    Small workloads are drawn on the host (numpy PCG64) so the oracle can
    regenerate them without a GPU; large ones on the device.
    """
    import torch
    qs, ks, dos = seq_shapes(w)
    on_host = small_on_host and w.S * w.H_q * w.D <= (1 << 26)
    if on_host:
        t = [host_tensor(qs, SEED_Q, w.dtype), host_tensor(ks, SEED_K, w.dtype),
             host_tensor(ks, SEED_V, w.dtype), host_tensor(dos, SEED_DO, w.dtype)]
        if device is not None:
            t = [x.to(device) for x in t]
        return t
    dev = device if device is not None else "cuda"
    return [device_tensor(qs, SEED_Q, w.dtype, dev), device_tensor(ks, SEED_K, w.dtype, dev),
            device_tensor(ks, SEED_V, w.dtype, dev), device_tensor(dos, SEED_DO, w.dtype, dev)]
