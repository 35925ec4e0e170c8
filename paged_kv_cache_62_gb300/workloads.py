"""Seeded synthetic decode workloads for the paged KV cache.

This module only *builds inputs*: sequence lengths, block tables, a physical
block pool filled with N(0, 1) bf16 values, query rows and the K/V rows of the
tokens a decode step appends.  It computes none of the operations under test
(no slot arithmetic, no store, no attention); both the CUDA library and the
CPU oracle consume what it returns.

Shapes follow the pages' models:

* Qwen3-0.6B: 28 layers, 16 query heads, 8 KV heads, head_dim 128, bf16
  (nano-vLLM lab manual §5.2.1; nano-vllm KV-cache post §1.3, §3.1).
* Qwen2.5-0.5B: 14 query heads, 2 KV heads, head_dim 64 (mini-vLLM README §1
  and §5 micro-benchmark shape).

Conventions (the plainest reading of the pages):

* ``context_lens[b]`` counts the token appended in this step (lab manual
  §5.2.1; KV-cache post §4.4), so that token sits at position ``L - 1``.
* Pool rows that no sequence owns hold a bf16 NaN canary; so does the row each
  appended token will be stored to, so a missed store or an over-read shows up
  as NaN downstream.
* A row of ``block_tables`` lists the sequence's physical block ids in logical
  order and is padded with -1 (MinivLLM review, decode branch).
* Prefix sharing (the long/mixed workload): the sequences of a group of 8 use
  the same physical ids for their leading *full* blocks, at most 64 of them;
  the block holding the appended token is always private (KV-cache post §3.4:
  only full blocks are shared; copy-on-write before a divergent write).

Randomness: structure (lengths, permutations, groups) comes from
``numpy.random.default_rng(seed)``; values come from a ``torch.Generator`` on
the target device seeded with the same number.  Draw order: lengths, shared
ids, block permutation, skipped token, then per layer q, K pool, V pool, new k,
new v.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 62000
BF16_NAN = float("nan")


@dataclass
class Spec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    layers: int = 1
    num_tokens: int | None = None          # kv_store rows (>= num_seqs); None = num_seqs
    description: str = ""


SPECS = {
    "tiny": Spec("tiny", 4, 4, 2, 64, 16, description=(
        "4 seqs, context_lens {1,15,17,40}, block_size 16, 4 q / 2 kv heads, head_dim 64, "
        "pool of 64 blocks by seeded permutation, kv_store of 4 tokens with one slot -1")),
    "qwen25_0p5b": Spec("qwen25_0p5b", 16, 14, 2, 64, 16, description=(
        "Qwen2.5-0.5B-shaped layer: batch 16, 14 q / 2 kv heads, head_dim 64, block_size 16, "
        "context_lens U[128,192], shuffled pool of 512 blocks")),
    "qwen3_0p6b": Spec("qwen3_0p6b", 64, 16, 8, 128, 256, description=(
        "Qwen3-0.6B-shaped layer: batch 64, 16 q / 8 kv heads, head_dim 128, block_size 256, "
        "context_lens U[512,4096], permuted pool sized 1.2x need")),
    "long_mixed": Spec("long_mixed", 256, 16, 8, 128, 16, description=(
        "batch 256, 16 q / 8 kv heads, head_dim 128, block_size 16, context_lens log-uniform "
        "[1,32768], groups of 8 seqs share their first 64 physical blocks")),
    "full_depth": Spec("full_depth", 128, 16, 8, 128, 256, layers=28, num_tokens=160, description=(
        "28 Qwen3-0.6B-shaped layers, batch 128, context_len 2048 each, block_size 256, "
        "kv_store slot_mapping padded with -1 to 160 rows")),
}
ORDER = ["tiny", "qwen25_0p5b", "qwen3_0p6b", "long_mixed", "full_depth"]


@dataclass
class Layer:
    q: torch.Tensor          # [B, Hq, D] bf16
    k_new: torch.Tensor      # [T, Hkv, D] bf16
    v_new: torch.Tensor      # [T, Hkv, D] bf16
    k_cache: torch.Tensor    # [NB, bs, Hkv, D] bf16
    v_cache: torch.Tensor    # [NB, bs, Hkv, D] bf16


@dataclass
class Workload:
    spec: Spec
    seed: int
    context_lens: torch.Tensor   # [B] int32
    block_tables: torch.Tensor   # [B, max_blocks] int32, -1 padded
    num_blocks: int
    skip_tokens: list            # token rows whose slot is forced to -1 (their KV is already resident)
    layers: list = field(default_factory=list)
    shared_blocks: int = 0       # physical blocks referenced by more than one sequence

    @property
    def num_tokens(self) -> int:
        return self.spec.num_tokens or self.spec.num_seqs

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def lens_host(self) -> np.ndarray:
        return self.context_lens.cpu().numpy()

    def kv_bytes_logical(self) -> int:
        """K+V bytes one decode call reads: sum_b L_b * Hkv * D * 2 bytes * 2 (K and V)."""
        s = self.spec
        return int(self.lens_host().astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2 * 2

    def kv_bytes_unique(self) -> int:
        """K+V bytes of the distinct (block, row) pairs one decode call reads."""
        s = self.spec
        lens = self.lens_host().astype(np.int64)
        bt = self.block_tables.cpu().numpy()
        rows = {}
        for b, L in enumerate(lens):
            nb = -(-int(L) // s.block_size)
            for i in range(nb):
                p = int(bt[b, i])
                rows[p] = max(rows.get(p, 0), min(s.block_size, int(L) - i * s.block_size))
        return int(sum(rows.values())) * s.num_kv_heads * s.head_dim * 2 * 2


def _lengths(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    n = spec.name
    if n == "tiny":
        return np.array([1, 15, 17, 40], np.int64)
    if n == "qwen25_0p5b":
        return rng.integers(128, 192, size=spec.num_seqs, endpoint=True)
    if n == "qwen3_0p6b":
        return rng.integers(512, 4096, size=spec.num_seqs, endpoint=True)
    if n == "long_mixed":
        u = rng.uniform(0.0, math.log(32768.0 + 1.0), size=spec.num_seqs)
        return np.clip(np.floor(np.exp(u)), 1, 32768).astype(np.int64)
    if n == "full_depth":
        return np.full(spec.num_seqs, 2048, np.int64)
    raise KeyError(n)


def _structure(spec: Spec, seed: int):
    """Lengths, block tables (physical ids), pool size, skipped tokens, and per-seq stored-row counts."""
    rng = np.random.default_rng(seed)
    lens = _lengths(spec, rng)
    bs = spec.block_size
    nblk = [-(-int(L) // bs) for L in lens]          # blocks each sequence references
    B = spec.num_seqs

    # Logical blocks that come from a group's shared prefix (long/mixed workload only).
    shared_count = np.zeros(B, np.int64)
    group_of = np.zeros(B, np.int64)
    if spec.name == "long_mixed":
        for b in range(B):
            group_of[b] = b // 8
            shared_count[b] = min(64, (int(lens[b]) - 1) // bs)
    n_groups = int(group_of.max()) + 1 if spec.name == "long_mixed" else 0
    shared_ids_needed = 64 * n_groups
    private_needed = sum(nblk[b] - int(shared_count[b]) for b in range(B))
    need = shared_ids_needed + private_needed

    if spec.name == "tiny":
        num_blocks = 64
    elif spec.name == "qwen25_0p5b":
        num_blocks = 512
    elif spec.name == "qwen3_0p6b":
        num_blocks = int(math.ceil(1.2 * need))
    else:
        num_blocks = need
    assert need <= num_blocks, (spec.name, need, num_blocks)

    perm = rng.permutation(num_blocks)
    cursor = 0
    shared_ids = []
    for _ in range(n_groups):
        shared_ids.append(perm[cursor:cursor + 64])
        cursor += 64
    max_blocks = max(nblk)
    bt = np.full((B, max_blocks), -1, np.int64)
    for b in range(B):
        k = int(shared_count[b])
        if k:
            bt[b, :k] = shared_ids[group_of[b]][:k]
        own = nblk[b] - k
        bt[b, k:nblk[b]] = perm[cursor:cursor + own]
        cursor += own

    skip = []
    if spec.name == "tiny":
        skip = [int(rng.integers(0, B))]
    return lens, bt, num_blocks, skip


def make(name: str, device="cpu", seed: int | None = None, layers: int | None = None) -> Workload:
    """Build the named workload on ``device`` (torch device string)."""
    spec = SPECS[name]
    if seed is None:
        seed = SEED_BASE + ORDER.index(name)
    lens, bt, num_blocks, skip = _structure(spec, seed)
    B, Hq, Hkv, D, bs = spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    T = spec.num_tokens or B
    n_layers = spec.layers if layers is None else layers

    # Rows of each physical block that hold cached tokens before this step.  A sequence owns
    # positions [0, L-1) of its blocks; the row of position L-1 is written by this step's store,
    # except for skipped tokens, whose row is already resident.
    filled = np.zeros(num_blocks, np.int64)
    refs = np.zeros(num_blocks, np.int64)
    for b in range(B):
        L = int(lens[b])
        resident = L if b in skip else L - 1
        nb = -(-L // bs)
        for i in range(nb):
            p = int(bt[b, i])
            refs[p] += 1
            covered = min(bs, max(0, resident - i * bs))
            filled[p] = max(filled[p], covered)

    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    row_ids = torch.arange(bs, device=dev).view(1, bs)
    canary = row_ids >= torch.as_tensor(filled, device=dev).view(num_blocks, 1)   # [NB, bs]

    def randn_bf16(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    wl = Workload(spec=spec, seed=seed,
                  context_lens=torch.as_tensor(lens, dtype=torch.int32, device=dev),
                  block_tables=torch.as_tensor(bt, dtype=torch.int32, device=dev),
                  num_blocks=num_blocks, skip_tokens=skip,
                  shared_blocks=int((refs > 1).sum()))
    for _ in range(n_layers):
        q = randn_bf16(B, Hq, D)
        kc = randn_bf16(num_blocks, bs, Hkv, D)
        kc[canary] = BF16_NAN
        vc = randn_bf16(num_blocks, bs, Hkv, D)
        vc[canary] = BF16_NAN
        kn = randn_bf16(T, Hkv, D)
        vn = randn_bf16(T, Hkv, D)
        wl.layers.append(Layer(q=q, k_new=kn, v_new=vn, k_cache=kc, v_cache=vc))
    return wl


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit pattern (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit pattern -> bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
