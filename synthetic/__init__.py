"""Seeded synthetic KV caches for the R-KV compression event.

This module only draws inputs: keys, values, window queries, sequence lengths
and block tables with the shapes and value structure of the five workloads
below. It holds none of the method's arithmetic, so both the CUDA library and
the CPU oracle can take their inputs from here without sharing any scoring,
selection or compaction code.

Workloads (shapes from the R-KV review page, "Installing R-KV and running a
first math evaluation": kv_budget 1024, window_size 8, mix_lambda 0.1,
divide_length 128; paged block size 16 from the hotdry.top blog, Ada-KV
section):

  0  one layer of a Llama-3-8B cache: 8 KV heads, 32 query heads, d=128,
     N = 1152 (budget 1024 + buffer 128), window 8, 25% near-duplicate tokens.
  1  all 32 Llama-3-8B layers, batch 1, same N; the near-duplicate fraction is
     drawn per layer from U[0.10, 0.40].
  2  batch 64, 32 layers, N = 2176 (budget 2048 + buffer 128); runs of 8-32
     repeated tokens cover 30% of each sequence.
  3  batch 16, 32 layers, N = 4352 (budget 4096 + buffer 256), window 16; keys
     drawn from 64 Gaussian clusters per head (spread 0.2).
  4  Qwen2-7B shape (28 layers, 4 KV heads, 28 query heads), batch 128, paged
     (block 16), N_b ~ U{1025..1152}; block tables deal a random permutation of
     a pool of 72 blocks per sequence.

Values are drawn in fp32 and rounded to bf16 (round to nearest even, torch's
conversion); both sides of every comparison see the same bf16 bytes.

Random streams: the structure (duplicate positions, run layout, lengths, block
tables) comes from numpy PCG64 streams keyed by (seed, layer); the float data
from a torch generator on the target device keyed the same way. Float values
therefore differ between a CPU and a CUDA generation of the same workload;
every comparison takes both sides' inputs from one generation.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SEED_BASE = 0x524B56  # per-workload seed = SEED_BASE + workload index


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    layers: int
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    budget: int
    buffer: int
    window: int
    mix_lambda: float
    keys: str                 # 'dups' | 'dups_layer' | 'runs' | 'clusters'
    dup_frac: float = 0.25    # for 'dups'
    paged: bool = False
    block_size: int = 16
    ragged: bool = False      # N_b ~ U{budget+1 .. budget+buffer}

    @property
    def max_seq_len(self) -> int:
        return self.budget + self.buffer

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def blocks_per_seq(self) -> int:
        return -(-self.max_seq_len // self.block_size)

    @property
    def events(self) -> int:
        return self.layers * self.batch


WORKLOADS = {
    0: Shape("llama8b-1layer-n1152", 1, 1, 8, 32, 128, 1024, 128, 8, 0.1, "dups"),
    1: Shape("llama3-8b-32layer-b1-n1152", 32, 1, 8, 32, 128, 1024, 128, 8, 0.1, "dups_layer"),
    2: Shape("llama8b-32layer-b64-n2176-runs", 32, 64, 8, 32, 128, 2048, 128, 8, 0.1, "runs"),
    3: Shape("llama8b-32layer-b16-n4352-clusters", 32, 16, 8, 32, 128, 4096, 256, 16, 0.1, "clusters"),
    4: Shape("qwen2-7b-28layer-b128-paged16-ragged", 28, 128, 4, 28, 128, 1024, 128, 8, 0.1, "dups",
             paged=True, ragged=True),
}


@dataclasses.dataclass
class Workload:
    shape: Shape
    seed: int
    k_cache: torch.Tensor            # contiguous [L][B][Hkv][Nmax][d] or paged pool [L][nblk][16][Hkv][d]
    v_cache: torch.Tensor
    q_window: torch.Tensor           # [L][B][Hq][w][d]
    seq_lens: torch.Tensor           # int32 [B]
    block_table: Optional[torch.Tensor]  # int32 [B][blocks_per_seq] (paged) or None
    num_blocks: int

    @property
    def events(self) -> int:
        return self.shape.events


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def _torch_gen(device: torch.device, seed: int, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    mixed = int(np.random.SeedSequence([seed, *key]).generate_state(1, dtype=np.uint64)[0])
    g.manual_seed(mixed & ((1 << 63) - 1))
    return g


def _dup_sources(rng: np.random.Generator, n: int, frac: float) -> np.ndarray:
    """Source index per position (-1 = fresh token): round(frac*n) positions in
    [1, n) without replacement, each a copy of a uniformly chosen earlier one."""
    src = np.full(n, -1, dtype=np.int64)
    count = int(round(frac * n))
    count = min(count, n - 1)
    if count <= 0:
        return src
    pos = rng.choice(np.arange(1, n), size=count, replace=False)
    src[pos] = (rng.random(count) * pos).astype(np.int64)  # uniform in [0, pos)
    return src


def _run_sources(rng: np.random.Generator, n: int, cover: float = 0.30,
                 rmin: int = 8, rmax: int = 32) -> np.ndarray:
    """Runs of r ~ U{rmin..rmax} copies of one earlier token, placed at random
    free offsets until at least cover*n positions are covered (the last run is
    cut to the remaining count)."""
    src = np.full(n, -1, dtype=np.int64)
    need = int(math.ceil(cover * n))
    covered = 0
    free = np.ones(n, dtype=bool)
    free[0] = False  # a run needs a source before it
    tries = 0
    while covered < need and tries < 100000:
        tries += 1
        r = int(rng.integers(rmin, rmax + 1))
        r = min(r, need - covered)
        start = int(rng.integers(1, n - r + 1))
        if not free[start:start + r].all():
            continue
        s = int(rng.integers(0, start))
        src[start:start + r] = s
        free[start:start + r] = False
        covered += r
    return src


def _chain_depth(src: np.ndarray) -> np.ndarray:
    """Depth of each position in its copy chain (0 for fresh tokens)."""
    depth = (src >= 0).astype(np.int64)
    while True:
        nd = np.where(src >= 0, depth[np.maximum(src, 0)] + 1, 0)
        if np.array_equal(nd, depth):
            return depth
        depth = nd


def _apply_copies(x: torch.Tensor, srcs: list, sigma: float, gen: torch.Generator) -> None:
    """x: fp32 [B][H][N][d]; row i of sequence b becomes row src[i] + N(0, sigma^2)
    noise (per head), resolved along copy chains in depth order."""
    B = x.shape[0]
    depths = [_chain_depth(s) for s in srcs]
    maxd = max((int(d.max()) for d in depths), default=0)
    for level in range(1, maxd + 1):
        bi, ii, jj = [], [], []
        for b in range(B):
            pos = np.nonzero(depths[b] == level)[0]
            bi.append(np.full(pos.size, b))
            ii.append(pos)
            jj.append(srcs[b][pos])
        bi = torch.from_numpy(np.concatenate(bi)).to(x.device)
        ii = torch.from_numpy(np.concatenate(ii)).to(x.device)
        jj = torch.from_numpy(np.concatenate(jj)).to(x.device)
        if bi.numel() == 0:
            continue
        noise = torch.randn((bi.numel(), x.shape[1], x.shape[3]), generator=gen,
                            device=x.device, dtype=torch.float32)
        x[bi, :, ii] = x[bi, :, jj] + sigma * noise


def generate(workload: int | Shape, *, layers: Optional[int] = None, batch: Optional[int] = None,
             device: str | torch.device = "cpu", seed: Optional[int] = None,
             seq_lens: Optional[np.ndarray] = None) -> Workload:
    """Draw one synthetic workload.

    `layers`/`batch` shrink a workload for tests that the oracle must finish in
    seconds (the per-layer and per-sequence structure is unchanged).
    `seq_lens` overrides the per-sequence lengths (each in [1, max_seq_len]).
    """
    if isinstance(workload, Shape):
        shape, widx = workload, 0
    else:
        shape, widx = WORKLOADS[workload], workload
    if layers is not None or batch is not None:
        shape = dataclasses.replace(shape, layers=layers or shape.layers, batch=batch or shape.batch)
    if seed is None:
        seed = SEED_BASE + widx
    device = torch.device(device)
    L, B, Hkv, Hq, d = shape.layers, shape.batch, shape.kv_heads, shape.q_heads, shape.head_dim
    Nmax, w = shape.max_seq_len, shape.window

    grng = _rng(seed, 1 << 20)
    if seq_lens is not None:
        lens = np.asarray(seq_lens, dtype=np.int64)
        assert lens.shape == (B,) and lens.min() >= 1 and lens.max() <= Nmax
    elif shape.ragged:
        lens = grng.integers(shape.budget + 1, shape.budget + shape.buffer + 1, size=B)
    else:
        lens = np.full(B, Nmax, dtype=np.int64)

    if shape.paged:
        nbps = shape.blocks_per_seq
        num_blocks = B * nbps
        perm = grng.permutation(num_blocks)
        table = perm.reshape(B, nbps).astype(np.int32)
        k_cache = torch.empty((L, num_blocks, shape.block_size, Hkv, d), dtype=torch.bfloat16, device=device)
        v_cache = torch.empty_like(k_cache)
    else:
        num_blocks = 0
        table = None
        k_cache = torch.empty((L, B, Hkv, Nmax, d), dtype=torch.bfloat16, device=device)
        v_cache = torch.empty_like(k_cache)
    q_window = torch.empty((L, B, Hq, w, d), dtype=torch.bfloat16, device=device)

    lam_rng = _rng(seed, 1 << 21)
    layer_frac = lam_rng.uniform(0.10, 0.40, size=L) if shape.keys == "dups_layer" else None

    for l in range(L):
        srng = _rng(seed, l)
        gen = _torch_gen(device, seed, l)
        k = torch.randn((B, Hkv, Nmax, d), generator=gen, device=device, dtype=torch.float32)
        if shape.keys == "clusters":
            centres = torch.randn((B, Hkv, 64, d), generator=gen, device=device, dtype=torch.float32)
            assign = torch.from_numpy(srng.integers(0, 64, size=(B, Hkv, Nmax))).to(device)
            k = torch.gather(centres, 2, assign[..., None].expand(B, Hkv, Nmax, d)) + 0.2 * k
            v = torch.randn((B, Hkv, Nmax, d), generator=gen, device=device, dtype=torch.float32)
        else:
            v = torch.randn((B, Hkv, Nmax, d), generator=gen, device=device, dtype=torch.float32)
            if shape.keys == "runs":
                srcs = [_run_sources(srng, int(lens[b])) for b in range(B)]
            else:
                frac = layer_frac[l] if layer_frac is not None else shape.dup_frac
                srcs = [_dup_sources(srng, int(lens[b]), frac) for b in range(B)]
            srcs = [np.concatenate([s, np.full(Nmax - s.size, -1, dtype=np.int64)]) for s in srcs]
            _apply_copies(k, srcs, 0.05, gen)
            _apply_copies(v, srcs, 0.05, gen)
        q = torch.randn((B, Hq, w, d), generator=gen, device=device, dtype=torch.float32)
        q_window[l] = q.to(torch.bfloat16)
        kb, vb = k.to(torch.bfloat16), v.to(torch.bfloat16)
        if shape.paged:
            tab = torch.from_numpy(table.astype(np.int64)).to(device).reshape(-1)
            bs = shape.block_size
            # logical [B][Hkv][Nmax][d] -> [B][nbps][bs][Hkv][d] -> pool blocks
            kl = kb.permute(0, 2, 1, 3).reshape(B, nbps, bs, Hkv, d).reshape(B * nbps, bs, Hkv, d)
            vl = vb.permute(0, 2, 1, 3).reshape(B, nbps, bs, Hkv, d).reshape(B * nbps, bs, Hkv, d)
            k_cache[l, tab] = kl
            v_cache[l, tab] = vl
        else:
            k_cache[l] = kb
            v_cache[l] = vb
        del k, v, kb, vb

    return Workload(
        shape=shape,
        seed=seed,
        k_cache=k_cache,
        v_cache=v_cache,
        q_window=q_window,
        seq_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        block_table=None if table is None else torch.from_numpy(table).to(device),
        num_blocks=num_blocks,
    )


def custom_shape(*, layers=1, batch=1, kv_heads=2, q_heads=4, head_dim=128, budget=64, buffer=16,
                 window=4, mix_lambda=0.1, keys="dups", dup_frac=0.25, paged=False, ragged=False) -> Shape:
    """A small ad-hoc shape for tests (same generator, any sizes)."""
    return Shape("custom", layers, batch, kv_heads, q_heads, head_dim, budget, buffer, window,
                 mix_lambda, keys, dup_frac=dup_frac, paged=paged, ragged=ragged)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def logical_rows(wl: Workload, cache: torch.Tensor, l: int, b: int, h: int, n: int) -> torch.Tensor:
    """The first n logical rows [n][d] of head h of sequence b in layer l."""
    if wl.block_table is None:
        return cache[l, b, h, :n]
    bs = wl.shape.block_size
    nb = -(-n // bs)
    blocks = wl.block_table[b, :nb].long()
    return cache[l, blocks, :, h].reshape(nb * bs, -1)[:n]
