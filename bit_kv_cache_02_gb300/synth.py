"""Seeded synthetic inputs and the workload shapes (no quantization or
attention arithmetic lives here).

The workloads stand in for the pages' Llama/Falcon/Mistral caches: keys and
values are N(0, 1) fp16 with a few fixed key channels per KV head scaled up
(the fixed-channel key outliers described in "KV cache quantization", "Keys
are harder than values"), queries are N(0, 1) fp16.  Both the CUDA path and
the CPU oracle receive exactly these tensors.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    seqs: int
    q_heads: int
    kv_heads: int
    ctx: int                 # prefilled tokens per sequence (max when ragged)
    bits: int
    ragged_min: int = 0      # > 0: per-sequence ctx drawn from U{ragged_min..ctx}
    num_sink: int = 0
    pre_rope: bool = False
    residual: int = 128
    outlier_channels_fixed: tuple = ()  # key channels scaled up, the same for every head ...
    n_outliers: int = 4      # ... or, when empty, this many drawn per (layer, KV head)
    outlier_mult: float = 15.0
    seed: int = 0
    decode_tokens: int = 1   # tokens appended before attending
    key_per_token: bool = False  # keys grouped per token (the ablation of per-channel keys)
    paged: bool = False      # group blocks in a shared pool behind a shuffled block table
    hadamard: bool = False   # tokens Walsh-Hadamard rotated before quantization
    dense_sparse: bool = False  # dense-and-sparse blocks (each slice's largest element kept in fp16)
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 1, 256, 2, outlier_channels_fixed=(3, 17, 64, 101),
                     outlier_mult=20.0,
                     decode_tokens=0),
    "llama2_7b_mha": Workload("llama2_7b_mha", 32, 16, 32, 32, 4096, 2),
    "llama3_8b_gqa_2bit": Workload("llama3_8b_gqa_2bit", 32, 64, 32, 8, 8192, 2, ragged_min=1024),
    "llama3_8b_gqa_4bit": Workload("llama3_8b_gqa_4bit", 32, 64, 32, 8, 8192, 4, ragged_min=1024),
    "long_1m": Workload("long_1m", 1, 1, 32, 32, 1 << 20, 2),
    "kvquant_prerope": Workload("kvquant_prerope", 32, 8, 32, 32, 16384, 2, num_sink=1, pre_rope=True),
    # the Llama-2 shape with keys grouped per token (ablation row)
    "llama2_7b_mha_key_per_token": Workload("llama2_7b_mha_key_per_token", 32, 16, 32, 32, 4096, 2,
                                            key_per_token=True),
    # the Llama-2 shape with its group blocks paged through a shuffled table
    "llama2_7b_mha_paged": Workload("llama2_7b_mha_paged", 32, 16, 32, 32, 4096, 2, paged=True),
    # the Llama-2 shape with Walsh-Hadamard rotated tokens, per-channel and per-token keys
    "llama2_7b_mha_hadamard": Workload("llama2_7b_mha_hadamard", 32, 16, 32, 32, 4096, 2, hadamard=True),
    "llama2_7b_mha_key_per_token_hadamard": Workload("llama2_7b_mha_key_per_token_hadamard", 32, 16, 32, 32,
                                                     4096, 2, key_per_token=True, hadamard=True),
    # the Llama-2 shape with dense-and-sparse blocks
    "llama2_7b_mha_outliers": Workload("llama2_7b_mha_outliers", 32, 16, 32, 32, 4096, 2,
                                       dense_sparse=True),
}


def context_lengths(w: Workload, layer_seed_offset: int = 0) -> np.ndarray:
    """Prefilled tokens per sequence (ragged workloads draw U{min..max})."""
    if w.ragged_min:
        rng = np.random.default_rng([w.seed, 7])
        return rng.integers(w.ragged_min, w.ctx + 1, size=w.seqs).astype(np.int32)
    return np.full(w.seqs, w.ctx, np.int32)


def block_table(w: Workload, layer: int, seqs: int, heads: int, max_groups: int) -> np.ndarray:
    """[seqs][heads][max_groups] int32: a seeded random assignment of the
    logical group blocks to the blocks of a pool of exactly that many."""
    rng = np.random.default_rng([w.seed, 13, layer])
    n = seqs * heads * max_groups
    return rng.permutation(n).astype(np.int32).reshape(seqs, heads, max_groups)


def outlier_channels(w: Workload, layer: int) -> np.ndarray:
    """[kv_heads][n] key channels scaled by outlier_mult in this layer."""
    if w.outlier_channels_fixed:
        return np.tile(np.array(w.outlier_channels_fixed, np.int64), (w.kv_heads, 1))
    rng = np.random.default_rng([w.seed, 11, layer])
    return np.stack([rng.choice(HEAD_DIM, w.n_outliers, replace=False) for _ in range(w.kv_heads)])


def kv_tokens(w: Workload, layer: int, tokens: int, seqs=None, heads=None, device="cpu", stream_id=0,
              token_offset: int = 0):
    """Keys and values [S][Hkv][tokens][D] fp16 of `layer`, tokens
    token_offset..token_offset+tokens-1 of each sequence's stream.

    Small requests are drawn with numpy on the host; `device` only decides
    where the result lives.  Requests of more than 2^26 elements are drawn
    with torch's generator on `device` (same seed -> same values on a given
    device type); `seqs`/`heads` select a subset for host-side checks.
    """
    S = w.seqs if seqs is None else len(seqs)
    H = w.kv_heads if heads is None else len(heads)
    shape = (w.seqs, w.kv_heads, tokens, HEAD_DIM)
    n = int(np.prod(shape))
    seed = [w.seed, layer, stream_id, token_offset]
    if n <= (1 << 26):
        rng = np.random.default_rng(seed)
        k = rng.standard_normal(shape, dtype=np.float32)
        v = rng.standard_normal(shape, dtype=np.float32)
        oc = outlier_channels(w, layer)
        for h in range(w.kv_heads):
            k[:, h, :, oc[h]] *= w.outlier_mult
        k = torch.from_numpy(k.astype(np.float16))
        v = torch.from_numpy(v.astype(np.float16))
        if seqs is not None:
            k, v = k[list(seqs)], v[list(seqs)]
        if heads is not None:
            k, v = k[:, list(heads)], v[:, list(heads)]
        return k.to(device), v.to(device)
    assert seqs is None and heads is None, "subsets of large draws come from slicing the full draw"
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.default_rng(seed).integers(1 << 62)))
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    oc = torch.as_tensor(outlier_channels(w, layer), device=device)
    for h in range(w.kv_heads):
        k[:, h, :, oc[h]] *= w.outlier_mult
    return k.half(), v.half()


def queries(w: Workload, layer: int, step: int = 0, device="cpu"):
    """Query [S][Hq][D] fp16 for decode step `step` of `layer`."""
    rng = np.random.default_rng([w.seed, layer, 99, step])
    q = rng.standard_normal((w.seqs, w.q_heads, HEAD_DIM), dtype=np.float32).astype(np.float16)
    return torch.from_numpy(q).to(device)
