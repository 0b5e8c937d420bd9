"""Seeded synthetic inputs of the hybrid-attention workloads.

This module only draws random tensors and lays them out; it computes none of the
method (no compression, no indexer score, no attention).  Both the CUDA path and
the CPU oracle consume the very tensors made here: large tensors are drawn on
the device that will hold them, and the oracle reads host copies of them.

Distributions (per workload): K, V, q ~ N(0,1)/sqrt(d); indexer keys and indexer
queries ~ N(0,1)/sqrt(d_I); indexer head weights ~ U(0,1); gate logits ~ N(0,1).
Values are drawn in float32 and rounded to the storage type (bfloat16 rounds to
nearest even).  Optional rotary embedding of the first `rope_dims` dims of q and
of the per-token keys (interleaved pairs (2i, 2i+1), frequency theta^(-2i/rope_dims),
angle = position * frequency) is part of making the inputs, before rounding.
Optional planting (million-token workload): a fraction of the CSA blocks of each
sequence get a component a*u_hat added to each of their per-token indexer keys,
u_hat = unit(sum_h w_h qI_h) of that sequence's decode query and a = plant_sigma /
sqrt(d_I), i.e. plant_sigma standard deviations of a per-token key's projection
onto u_hat.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "csa" or "hca"
    B: int               # sequences
    L: int               # tokens in the cache, including the query tokens
    H: int
    d: int
    n_win: int
    m: int
    k: int               # top-k (CSA)
    H_I: int
    d_I: int
    dtype: str           # "f32" or "bf16"
    Tq: int = 1          # queries per sequence (1 = decode; else a prefill chunk at the end)
    rope_dims: int = 0
    rope_theta: float = 10000.0
    plant_frac: float = 0.0
    plant_sigma: float = 0.0
    seed: int = 0
    fmt: int = 0         # storage-format bits of the layer (2: FP4 indexer, bfloat16 scores)

    @property
    def n_blocks(self) -> int:
        return self.L // self.m

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def decode(self) -> bool:
        return self.Tq == 1

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # tiny fp32 layers: 1 sequence, 1024 tokens, 1 decode query
    "tiny_csa": Workload("tiny_csa", "csa", 1, 1024, 8, 64, 128, 4, 16, 2, 32, "f32"),
    "tiny_hca": Workload("tiny_hca", "hca", 1, 1024, 8, 64, 128, 128, 16, 2, 32, "f32"),
    # CSA decode: 32 sequences at 65,536 tokens, RoPE on the first 64 dims
    "csa_decode_64k": Workload("csa_decode_64k", "csa", 32, 65536, 64, 512, 128, 4, 512, 64, 128,
                               "bf16", rope_dims=64),
    # HCA decode: 32 sequences at 131,072 tokens
    "hca_decode_128k": Workload("hca_decode_128k", "hca", 32, 131072, 64, 512, 128, 128, 512, 64,
                                128, "bf16"),
    # CSA prefill: 4,096 new tokens after 131,072 cached tokens
    "csa_prefill_4k": Workload("csa_prefill_4k", "csa", 1, 131072 + 4096, 64, 512, 128, 4, 512,
                               64, 128, "bf16", Tq=4096),
    # million-token decode, both layer kinds
    "csa_decode_1m": Workload("csa_decode_1m", "csa", 4, 1 << 20, 128, 512, 128, 4, 1024, 64, 128,
                              "bf16", plant_frac=0.01, plant_sigma=3.0),
    "hca_decode_1m": Workload("hca_decode_1m", "hca", 4, 1 << 20, 128, 512, 128, 128, 1024, 64,
                              128, "bf16"),
}
# the same CSA decodes with the indexer in FP4 and bfloat16 index scores
WORKLOADS["csa_decode_64k_fp4"] = replace(WORKLOADS["csa_decode_64k"], name="csa_decode_64k_fp4",
                                          fmt=2)
WORKLOADS["csa_decode_1m_fp4"] = replace(WORKLOADS["csa_decode_1m"], name="csa_decode_1m_fp4",
                                         fmt=2)
# compressed K/V in the FP8 format (RoPE dims bfloat16, the rest e4m3), and both formats
WORKLOADS["csa_decode_64k_kv8"] = replace(WORKLOADS["csa_decode_64k"], name="csa_decode_64k_kv8",
                                          fmt=1)
WORKLOADS["hca_decode_128k_kv8"] = replace(WORKLOADS["hca_decode_128k"],
                                           name="hca_decode_128k_kv8", fmt=1)
WORKLOADS["csa_decode_1m_fp4_kv8"] = replace(WORKLOADS["csa_decode_1m"],
                                             name="csa_decode_1m_fp4_kv8", fmt=3)

_TENSOR_IDS = {"k_tok": 1, "v_tok": 2, "ki_tok": 3, "gate": 4, "q": 5, "qI": 6, "w": 7,
               "plant": 8, "extra": 9}


def _gen(device, seed: int, tensor: str, part: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _TENSOR_IDS[tensor] * 7919 + part) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _normal(shape, std, device, seed, tensor, part=0):
    g = _gen(device, seed, tensor, part)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _rope_(x: torch.Tensor, pos: torch.Tensor, dims: int, theta: float):
    """Rotate the first `dims` dims of x[..., pos_axis, :] in place (float32)."""
    i = torch.arange(dims // 2, device=x.device, dtype=torch.float64)
    freq = theta ** (-2.0 * i / dims)
    ang = pos.to(torch.float64)[..., None] * freq                 # [..., dims/2]
    c, s = torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)
    a, b = x[..., 0:dims:2].clone(), x[..., 1:dims:2].clone()
    x[..., 0:dims:2] = a * c - b * s
    x[..., 1:dims:2] = a * s + b * c


def query_positions(w: Workload, device) -> torch.Tensor:
    """int32 [B, Tq]: absolute positions of the queries (the last Tq tokens)."""
    pos = torch.arange(w.L - w.Tq, w.L, dtype=torch.int32, device=device)
    return pos.repeat(w.B, 1).contiguous()


def make_tokens(w: Workload, device) -> dict:
    """Per-token caches: k_tok, v_tok [B, L, d], ki_tok [B, L, d_I] (CSA), gate [B, L]."""
    dt = w.torch_dtype
    out = {"k_tok": torch.empty((w.B, w.L, w.d), dtype=dt, device=device),
           "v_tok": torch.empty((w.B, w.L, w.d), dtype=dt, device=device),
           "gate": torch.empty((w.B, w.L), dtype=torch.float32, device=device)}
    if w.kind == "csa":
        out["ki_tok"] = torch.empty((w.B, w.L, w.d_I), dtype=dt, device=device)
    chunk = 1 << 17                                               # tokens per draw
    for b in range(w.B):
        for c0 in range(0, w.L, chunk):
            c1 = min(w.L, c0 + chunk)
            part = b * 4096 + c0 // chunk
            kk = _normal((c1 - c0, w.d), 1 / math.sqrt(w.d), device, w.seed, "k_tok", part)
            if w.rope_dims:
                _rope_(kk, torch.arange(c0, c1, device=device), w.rope_dims, w.rope_theta)
            out["k_tok"][b, c0:c1] = kk.to(dt)
            out["v_tok"][b, c0:c1] = _normal((c1 - c0, w.d), 1 / math.sqrt(w.d), device, w.seed,
                                             "v_tok", part).to(dt)
            out["gate"][b, c0:c1] = _normal((c1 - c0,), 1.0, device, w.seed, "gate", part)
            if w.kind == "csa":
                out["ki_tok"][b, c0:c1] = _normal((c1 - c0, w.d_I), 1 / math.sqrt(w.d_I), device,
                                                  w.seed, "ki_tok", part).to(dt)
    return out


def make_queries(w: Workload, device) -> dict:
    """q [B, Tq, H, d]; for CSA also qI [B, Tq, H_I, d_I] and w_idx [B, Tq, H_I]."""
    dt = w.torch_dtype
    q = _normal((w.B, w.Tq, w.H, w.d), 1 / math.sqrt(w.d), device, w.seed, "q")
    if w.rope_dims:
        pos = query_positions(w, device)[:, :, None].expand(w.B, w.Tq, w.H)
        _rope_(q, pos, w.rope_dims, w.rope_theta)
    out = {"q": q.to(dt).contiguous(), "q_pos": query_positions(w, device),
           "ctx_len": torch.full((w.B,), w.L, dtype=torch.int32, device=device)}
    if w.kind == "csa":
        out["qI"] = _normal((w.B, w.Tq, w.H_I, w.d_I), 1 / math.sqrt(w.d_I), device, w.seed,
                            "qI").to(dt).contiguous()
        g = _gen(device, w.seed, "w", 0)
        out["w_idx"] = torch.rand((w.B, w.Tq, w.H_I), generator=g, device=device,
                                  dtype=torch.float32)
    return out


def plant_blocks(w: Workload, tokens: dict, queries: dict, n_eligible_blocks: int) -> torch.Tensor:
    """Add the planted component to a fraction of the CSA blocks (in place).

    Returns int64 [B, n_plant]: the planted block indices of each sequence, sorted.
    Only blocks below `n_eligible_blocks` are chosen, so every planted block is
    visible to the decode query.
    """
    n_plant = int(round(w.plant_frac * w.n_blocks))
    device = tokens["ki_tok"].device
    dt = w.torch_dtype
    planted = []
    for b in range(w.B):
        g = _gen(device, w.seed, "plant", b)
        blocks = torch.randperm(n_eligible_blocks, generator=g, device=device)[:n_plant]
        blocks, _ = torch.sort(blocks)
        u = (queries["w_idx"][b, -1, :, None].to(torch.float32)
             * queries["qI"][b, -1].to(torch.float32)).sum(0)
        u_hat = u / u.norm()
        amp = w.plant_sigma / math.sqrt(w.d_I)
        rows = (blocks[:, None] * w.m + torch.arange(w.m, device=device)).reshape(-1)
        ki = tokens["ki_tok"][b].index_select(0, rows).to(torch.float32) + amp * u_hat
        tokens["ki_tok"][b].index_copy_(0, rows, ki.to(dt))
        planted.append(blocks)
    return torch.stack(planted)


def random_index_sets(B: int, Tq: int, k: int, n_valid: torch.Tensor, device, seed: int,
                      pad_frac: float = 0.0) -> torch.Tensor:
    """int32 [B, Tq, k]: distinct ascending indices below n_valid[b, t] (then -1 padding).

    A generator-made stand-in for a top-k result, for testing the attention call
    on its own.
    """
    out = torch.full((B, Tq, k), -1, dtype=torch.int32)
    g = torch.Generator().manual_seed(seed)
    nv = n_valid.to("cpu").reshape(B, Tq)
    for b in range(B):
        for t in range(Tq):
            n = int(nv[b, t])
            take = min(k, n)
            take = take - int(round(pad_frac * take))
            if take <= 0:
                continue
            sel = torch.randperm(n, generator=g)[:take].sort().values
            out[b, t, :take] = sel.to(torch.int32)
    return out.to(device)


def gaussian(shape, device, seed: int, std: float = 1.0, dtype=torch.float32, part: int = 0):
    """Generic seeded Gaussian tensor (test fixtures)."""
    return _normal(shape, std, device, seed, "extra", part).to(dtype)
