"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and
the benchmark.

This module draws random numbers and fixes shapes; it holds none of the
method's arithmetic (no compression, scoring, selection or attention).

Recipe (every workload): one ``torch.Generator`` seeded per workload; floating
tensors are drawn in fp32 (``randn`` = N(0,1), ``rand`` = U(0,1)) and then
rounded to the workload dtype with round-to-nearest-even; integer draws use
``randint``.  Draw order is fixed per builder (listed in each docstring).  The
same seed gives different numbers on a CPU and a CUDA generator, so a run
draws every tensor on ONE device and hands copies of those very tensors to
both sides.

Shapes follow the five settings the method is measured on:
  csa_tiny       T=2048, Q[T,8,64], K,V[T,64], G[4,64], indexer 4x32, k=32,
                 W=64, fp32, seed 0
  csa_prefill    T=32768, Q[T,64,128], K,V[T,128], G[4,128], indexer 8x64,
                 k=512, W=128, bf16, seed 1
  hca_prefill    T=131072, Q[T,64,128], K,V[T,128], G'[128,128], W=128, bf16,
                 seed 2
  csa_decode     B=64, ctx ~ U[65536, 262144], Q[64,128,128], compressed
                 cache [ctx/4,128], indexer keys [ctx/4,8,64], k=1024, W=128,
                 bf16, seed 3
  layer_pair_1m  context 1,048,576, last 4096 positions queried; a CSA layer
                 (m=4, indexer 8x64, k=1024, W=128) and an HCA layer (m'=128,
                 W=128), Q[4096,128,128] each, own raw K,V[1M,128] each, bf16,
                 seed 4
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Batch:
    """Ragged batch layout (host copies).  Sequence b owns query rows
    cu_q[b]..cu_q[b+1]-1 at consecutive absolute positions starting at
    q_pos0[b]; compressed entries cu_c[b]..cu_c[b+1]-1 (sequence-local entry j
    is row cu_c[b]+j); raw rows cu_raw[b]..cu_raw[b+1]-1 holding positions
    raw_pos0[b], raw_pos0[b]+1, ..."""
    cu_q: list
    q_pos0: list
    cu_c: list
    cu_raw: list
    raw_pos0: list

    @property
    def B(self) -> int:
        return len(self.q_pos0)

    def positions(self):
        """Absolute position of every query row (a plain list of ints)."""
        out = []
        for b in range(self.B):
            out.extend(range(self.q_pos0[b], self.q_pos0[b] + self.cu_q[b + 1] - self.cu_q[b]))
        return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(g: torch.Generator, shape, dtype: str, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def uniform(g: torch.Generator, shape, dtype: str, device) -> torch.Tensor:
    x = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def single(T_raw: int, q_pos0: int, Nq: int, Tc: int, raw_pos0: int = 0) -> Batch:
    return Batch(cu_q=[0, Nq], q_pos0=[q_pos0], cu_c=[0, Tc], cu_raw=[0, T_raw],
                 raw_pos0=[raw_pos0])


def csa_layer(*, T: int, H: int, d: int, HI: int, dI: int, m: int, k: int, W: int,
              dtype: str, seed: int, device="cpu", q_from: int = 0) -> Dict:
    """One CSA layer over one sequence of T raw tokens, querying positions
    q_from..T-1.  Draw order: Q, K, V, G (used as both G_K and G_V), q_I, k_I
    (one per full block, floor(T/m) rows), w.  Gate logits and head weights
    are fp32 whatever the dtype."""
    g = _gen(seed, device)
    Nq = T - q_from
    Tc = T // m
    out = dict(kind="csa", T=T, H=H, d=d, HI=HI, dI=dI, m=m, k=k, W=W, dtype=dtype,
               scale=1.0 / math.sqrt(d), seed=seed)
    out["Q"] = normal(g, (Nq, H, d), dtype, device)
    out["K"] = normal(g, (T, d), dtype, device)
    out["V"] = normal(g, (T, d), dtype, device)
    out["G"] = normal(g, (m, d), "f32", device)
    out["qI"] = normal(g, (Nq, HI, dI), dtype, device)
    out["kI"] = normal(g, (Tc, HI, dI), dtype, device)
    out["w"] = uniform(g, (Nq, HI), "f32", device)
    out["batch"] = single(T, q_from, Nq, Tc)
    return out


def csa_layer_token_gated(*, T: int, H: int, d: int, HI: int, dI: int, m: int, k: int, W: int,
                          dtype: str, seed: int, device="cpu", q_from: int = 0,
                          gate_scale: float = 1.0) -> Dict:
    """A CSA layer whose compressor gates come from each token: per-token gate
    logits Z_K, Z_V [T, d] and token-level indexer keys kI_tok [T, HI, dI]
    with their own gate logits Z_I [T, HI, dI] (the indexer-side compressor).
    Gate logits are N(0, gate_scale^2), the distribution of a random
    projection of random hidden states.  Draw order: Q, K, V, Z_K, Z_V, q_I,
    kI_tok, Z_I, w.  No compressed tensor is drawn: both sides compress."""
    g = _gen(seed, device)
    Nq = T - q_from
    out = dict(kind="csa_token_gated", T=T, H=H, d=d, HI=HI, dI=dI, m=m, k=k, W=W,
               dtype=dtype, scale=1.0 / math.sqrt(d), seed=seed)
    out["Q"] = normal(g, (Nq, H, d), dtype, device)
    out["K"] = normal(g, (T, d), dtype, device)
    out["V"] = normal(g, (T, d), dtype, device)
    out["ZK"] = normal(g, (T, d), "f32", device) * gate_scale
    out["ZV"] = normal(g, (T, d), "f32", device) * gate_scale
    out["qI"] = normal(g, (Nq, HI, dI), dtype, device)
    out["kI_tok"] = normal(g, (T, HI, dI), dtype, device)
    out["ZI"] = normal(g, (T, HI, dI), "f32", device) * gate_scale
    out["w"] = uniform(g, (Nq, HI), "f32", device)
    out["batch"] = single(T, q_from, Nq, T // m)
    return out


def hca_layer(*, T: int, H: int, d: int, m: int, W: int, dtype: str, seed: int,
              device="cpu", q_from: int = 0) -> Dict:
    """One HCA layer over one sequence.  Draw order: Q, K, V, G'."""
    g = _gen(seed, device)
    Nq = T - q_from
    out = dict(kind="hca", T=T, H=H, d=d, m=m, W=W, dtype=dtype, scale=1.0 / math.sqrt(d),
               seed=seed)
    out["Q"] = normal(g, (Nq, H, d), dtype, device)
    out["K"] = normal(g, (T, d), dtype, device)
    out["V"] = normal(g, (T, d), dtype, device)
    out["G"] = normal(g, (m, d), "f32", device)
    out["batch"] = single(T, q_from, Nq, T // m)
    return out


def csa_decode(*, B: int, ctx_lo: int, ctx_hi: int, H: int, d: int, HI: int, dI: int,
               m: int, k: int, W: int, dtype: str, seed: int, device="cpu") -> Dict:
    """Batch of B sequences with one query each at position ctx_b - 1.
    Draw order: ctx lengths (randint, inclusive range, first because they fix
    every other shape), Q, compressed Kc, Vc (sum of floor(ctx_b/m) rows),
    raw window K, V (the last W positions of each sequence), q_I, k_I, w."""
    g = _gen(seed, device)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g, device=device).tolist()
    Tcs = [c // m for c in ctx]
    cu_c = [0]
    for t in Tcs:
        cu_c.append(cu_c[-1] + t)
    nraw = [min(W, c) for c in ctx]
    cu_raw = [0]
    for n in nraw:
        cu_raw.append(cu_raw[-1] + n)
    batch = Batch(cu_q=list(range(B + 1)), q_pos0=[c - 1 for c in ctx], cu_c=cu_c,
                  cu_raw=cu_raw, raw_pos0=[c - n for c, n in zip(ctx, nraw)])
    out = dict(kind="csa_decode", B=B, ctx=ctx, H=H, d=d, HI=HI, dI=dI, m=m, k=k, W=W,
               dtype=dtype, scale=1.0 / math.sqrt(d), seed=seed, batch=batch)
    out["Q"] = normal(g, (B, H, d), dtype, device)
    out["Kc"] = normal(g, (cu_c[-1], d), dtype, device)
    out["Vc"] = normal(g, (cu_c[-1], d), dtype, device)
    out["Kraw"] = normal(g, (cu_raw[-1], d), dtype, device)
    out["Vraw"] = normal(g, (cu_raw[-1], d), dtype, device)
    out["qI"] = normal(g, (B, HI, dI), dtype, device)
    out["kI"] = normal(g, (cu_c[-1], HI, dI), dtype, device)
    out["w"] = uniform(g, (B, HI), "f32", device)
    return out


def ragged(layers, keys) -> Dict:
    """A ragged batch made of single-sequence workloads (each from csa_layer,
    csa_layer_token_gated or hca_layer, in the given order): the tensors named
    in ``keys`` are concatenated along their first (row) axis and the batch
    arrays are offset accordingly.  The per-sequence workloads are kept under
    "parts" so that a check can slice each sequence back out."""
    cu_q, q_pos0, cu_c, cu_raw, raw_pos0 = [0], [], [0], [0], []
    for L in layers:
        b = L["batch"]
        cu_q.append(cu_q[-1] + b.cu_q[1] - b.cu_q[0])
        q_pos0.append(b.q_pos0[0])
        cu_c.append(cu_c[-1] + b.cu_c[1] - b.cu_c[0])
        cu_raw.append(cu_raw[-1] + b.cu_raw[1] - b.cu_raw[0])
        raw_pos0.append(b.raw_pos0[0])
    out = {key: val for key, val in layers[0].items() if not isinstance(val, torch.Tensor)}
    for key in keys:
        out[key] = torch.cat([L[key] for L in layers], dim=0)
    out["batch"] = Batch(cu_q=cu_q, q_pos0=q_pos0, cu_c=cu_c, cu_raw=cu_raw,
                         raw_pos0=raw_pos0)
    out["parts"] = list(layers)
    return out


def layer_pair(*, ctx: int = 1 << 20, chunk: int = 4096, H: int = 128, d: int = 128,
               HI: int = 8, dI: int = 64, m_csa: int = 4, m_hca: int = 128, k: int = 1024,
               W: int = 128, dtype: str = "bf16", seed: int = 4, device="cpu") -> Dict:
    """Interleaved CSA + HCA layer pair over a context of ``ctx`` tokens whose
    last ``chunk`` positions are queried.  Each layer has its own raw K, V over
    the whole context; the compressed entries of the positions before the
    chunk are the compressor's output on that prefix (a set-up step of each
    side).  Draw order: CSA (Q, K, V, G, q_I, k_I over all ctx/m entries, w),
    then HCA (Q, K, V, G')."""
    csa = csa_layer(T=ctx, H=H, d=d, HI=HI, dI=dI, m=m_csa, k=k, W=W, dtype=dtype,
                    seed=seed, device=device, q_from=ctx - chunk)
    hca = hca_layer(T=ctx, H=H, d=d, m=m_hca, W=W, dtype=dtype, seed=seed + 1000,
                    device=device, q_from=ctx - chunk)
    return dict(kind="layer_pair", ctx=ctx, chunk=chunk, csa=csa, hca=hca, dtype=dtype)


# The five measured settings, by name.
CONFIGS = {
    "csa_tiny": lambda device="cpu": csa_layer(T=2048, H=8, d=64, HI=4, dI=32, m=4, k=32,
                                               W=64, dtype="f32", seed=0, device=device),
    "csa_prefill": lambda device="cpu": csa_layer(T=32768, H=64, d=128, HI=8, dI=64, m=4,
                                                  k=512, W=128, dtype="bf16", seed=1,
                                                  device=device),
    "hca_prefill": lambda device="cpu": hca_layer(T=131072, H=64, d=128, m=128, W=128,
                                                  dtype="bf16", seed=2, device=device),
    "csa_decode": lambda device="cpu": csa_decode(B=64, ctx_lo=65536, ctx_hi=262144, H=128,
                                                  d=128, HI=8, dI=64, m=4, k=1024, W=128,
                                                  dtype="bf16", seed=3, device=device),
    "layer_pair_1m": lambda device="cpu": layer_pair(device=device),
}
