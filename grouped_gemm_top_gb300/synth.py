"""Seeded synthetic inputs for the MoE layer (shared by tests, bench and the
smoke run).  Holds no step of the method: only random draws with the shapes
and distributions of the workloads.

Recipe (per tensor, one torch.Generator seeded with the tensor's seed, on the
device the tensor is made on):
  logits  fp32 [T, E] ~ N(0, 1)                               seed 0
          optional Zipf(s) popularity bias -s*ln(rank_e), rank a seeded
          permutation of 1..E (numpy, seed + 7919)
  x       bf16 [T, d] ~ N(0, 1)                               seed 1
  W1      bf16 [E, d, 2f] ~ N(0, 0.02^2)                      seed 2
  W2      bf16 [E, f, d]  ~ N(0, 0.02^2)                      seed 3
  dout    bf16 [T, d] ~ N(0, 1)                               seed 4
Large tensors are drawn one expert (or 64M elements) at a time so no fp32
copy of a whole weight is ever held.
"""
from __future__ import annotations

import numpy as np
import torch

SEED_LOGITS, SEED_X, SEED_W1, SEED_W2, SEED_DOUT = 0, 1, 2, 3, 4


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """-s * ln(rank_e) with rank a seeded random permutation of 1..E."""
    rank = np.random.default_rng(seed + 7919).permutation(E) + 1
    return (-s * np.log(rank)).astype(np.float32)


def make_logits(T, E, seed=SEED_LOGITS, device="cpu", zipf_s=None):
    g = _gen(seed, device)
    out = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if zipf_s:
        out += torch.from_numpy(zipf_bias(E, zipf_s, seed)).to(device)
    return out


def make_normal_bf16(shape, seed, device="cpu", std=1.0, chunk_elems=1 << 26):
    """bf16 tensor of N(0, std^2) draws, generated in chunks along dim 0."""
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    per_row = flat.shape[1]
    rows = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        blk = torch.randn((r1 - r0, per_row), generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            blk.mul_(std)
        flat[r0:r1].copy_(blk)
    return out


def make_layer_inputs(T, d, E, f, device="cpu", zipf_s=None, seed_offset=0, weights=True, w_std=0.02, n_shared=0):
    """Router logits [T, E], x and dout [T, d] (bf16, N(0, 1)) and, with
    weights, W1 [E+S, d, 2f] and W2 [E+S, f, d] (bf16, N(0, w_std^2); the S
    shared experts' weights last)."""
    inp = dict(
        logits=make_logits(T, E, SEED_LOGITS + seed_offset, device, zipf_s),
        x=make_normal_bf16((T, d), SEED_X + seed_offset, device),
        dout=make_normal_bf16((T, d), SEED_DOUT + seed_offset, device),
    )
    if weights:
        inp["W1"] = make_normal_bf16((E + n_shared, d, 2 * f), SEED_W1, device, std=w_std)
        inp["W2"] = make_normal_bf16((E + n_shared, f, d), SEED_W2, device, std=w_std)
    return inp


def dirichlet_group_sizes(G: int, M: int, alpha: float, seed: int) -> np.ndarray:
    """Split M rows into G groups: p ~ Dirichlet(alpha), m_g = floor(p_g M),
    then +1 to the largest remainders until the sizes sum to M."""
    p = np.random.default_rng(seed).dirichlet(np.full(G, alpha))
    raw = p * M
    m = np.floor(raw).astype(np.int64)
    short = M - int(m.sum())
    order = np.argsort(-(raw - m), kind="stable")
    m[order[:short]] += 1
    return m
