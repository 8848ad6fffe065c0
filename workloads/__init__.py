"""Seeded synthetic workloads for the paged KV cache (shared by tests and bench).

This module is the ONLY code both the oracle side and the CUDA side consume. It
holds shapes, seeds, random draws and the order of host operations -- none of
the method's arithmetic (no slot, table, softmax or copy logic lives here).
Every random number the method needs (the initial free-queue order, the churn
of dummy allocations, K/V/q values) is drawn here and passed in as input.

Five workloads, shaped like the pages' serving cases (7B and 13B head shapes,
mixed context lengths, a shared system prompt); no public dataset is involved:

1. tiny    -- 1 layer, 4 heads x 64, B=16, 64 blocks, 4 sequences of
              {17, 33, 50, 64} tokens; one append + one attention step.
2. 7b      -- 32 layers, 32 heads x 128, B=16, 32 sequences of U[256, 2048]
              tokens, pool = 1.3 x the blocks needed, shuffled block ids.
3. prefix  -- 7B shape, B=16, 64 sequences forked from one 520-token prompt
              (33 shared blocks), then per-request suffixes of U[64, 512]
              tokens written through the append path (the first one
              copy-on-writes the shared partial block), then decode steps.
4. 13b     -- 40 layers, 40 heads x 128, B=32, 128 sequences, lengths
              lognormal(median 300, sigma 1.034) clipped to [16, 4096]; the
              pool ends 90 % occupied after a seeded alloc/free churn of dummy
              sequences interleaved with the batch's admissions.
5. long    -- 7B heads, B=256 (4 MiB per page per layer), 16 sequences of
              U[4096, 16384] tokens; the block-size sweep re-runs it at
              B = 8/16/32/64 with identical per-token data.

Values: K, V, q, new-token K/V are fp16 draws of N(0, 1). Seed = 1000 + index.

A workload's ``script`` is a list of host operations, each a tuple:

* ``("admit", s, T)``        sequence s starts with T tokens in fresh blocks;
* ``("fork", src, dst)``     sequence dst shares every block of src;
* ``("dummy_alloc", d, n)``  an unrelated request d takes n blocks;
* ``("dummy_free", d)``      request d releases its blocks;
* ``("write", counts)``      counts[s] new tokens of sequence s are appended
                              (data from :func:`write_values`);
* ``("prompt", s, tokens)``  sequence s arrives with prompt token ids ``tokens``:
                              its leading full blocks are looked up in the prefix
                              cache, the rest is written (data from
                              :func:`write_values`) and its full blocks registered.

Workload 3 comes in two forms: ``prefix_mode="fork"`` (the shared prompt is
forked to every request, the first suffix token copies the shared partial
block) and ``prefix_mode="hash"`` (every request arrives with the same 520
prompt tokens plus its own suffix tokens and finds the shared blocks through
the prefix cache).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

CONFIG_NAMES = {1: "tiny", 2: "7b", 3: "prefix", 4: "13b", 5: "long"}


@dataclasses.dataclass
class Workload:
    index: int
    name: str
    num_layers: int
    num_heads: int
    head_dim: int
    block_size: int
    num_seqs: int
    num_blocks: int
    max_blocks: int
    context_lens: np.ndarray          # int32 [S], lengths after the setup script
    free_order: np.ndarray            # int32 [N], initial free-queue order
    script: list
    decode_steps: int
    seed: int
    layout: str = "HND"
    description: str = ""
    kv_dtype: str = "f16"

    @property
    def kv_bytes_per_token_layer(self) -> int:
        """Bytes of K and V one token holds in one layer (E4M3: codes plus the two row scales)."""
        if self.kv_dtype == "e4m3":
            return 2 * self.num_heads * (self.head_dim + 4)
        return 2 * self.num_heads * self.head_dim * 2

    def describe(self) -> dict:
        return {
            "workload": f"cfg{self.index}-{self.name}",
            "layers": self.num_layers, "heads": self.num_heads, "head_dim": self.head_dim,
            "block_size": self.block_size, "batch": self.num_seqs, "pool_blocks": self.num_blocks,
            "mean_context": float(np.mean(self.context_lens)) if self.num_seqs else 0.0,
            "layout": self.layout, "kv_dtype": self.kv_dtype,
        }


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(t) for t in tags]))


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _finish(index, name, L, H, D, B, lens, script, steps, seed, N, layout, desc, extra_tokens=0):
    lens = np.asarray(lens, dtype=np.int32)
    tmax = int(lens.max()) if lens.size else 0
    max_blocks = max(1, _ceil_div(tmax + steps + extra_tokens + 1, B))
    order = _rng(seed, 7).permutation(N).astype(np.int32)
    return Workload(index=index, name=name, num_layers=L, num_heads=H, head_dim=D, block_size=B,
                    num_seqs=len(lens), num_blocks=int(N), max_blocks=int(max_blocks),
                    context_lens=lens, free_order=order, script=script, decode_steps=int(steps),
                    seed=int(seed), layout=layout, description=desc)


def make_workload(index: int, *, kv_dtype: str = "f16", **kw) -> Workload:
    """The seeded workload ``index`` (1..5); keyword overrides shrink it for tests.

    ``len_scale`` multiplies sampled context lengths (tests use it to keep the
    oracle fast while keeping the length mix). ``kv_dtype`` "e4m3" asks for a
    quantised cache (the pools then start with random finite E4M3 codes and
    scales instead of fp16 draws).
    """
    w = _make_workload(index, **kw)
    w.kv_dtype = kv_dtype
    return w


def _make_workload(index: int, *, num_layers: Optional[int] = None, num_seqs: Optional[int] = None,
                   block_size: Optional[int] = None, decode_steps: Optional[int] = None,
                   layout: str = "HND", seed: Optional[int] = None,
                   len_scale: float = 1.0, prefix_mode: str = "fork") -> Workload:
    seed = 1000 + index if seed is None else seed
    r = _rng(seed, 1)
    if index == 1:
        L, H, D, B = 1, 4, 64, 16
        lens = [17, 33, 50, 64]
        S = len(lens) if num_seqs is None else num_seqs
        lens = lens[:S]
        B = block_size or B
        steps = 1 if decode_steps is None else decode_steps
        N = 64
        script = [("admit", s, int(t)) for s, t in enumerate(lens)]
        return _finish(1, "tiny", num_layers or L, H, D, B, lens, script, steps, seed, N, layout,
                       "1 layer, 4x64 heads, B=16, 64 blocks, lens {17,33,50,64}")
    if index == 2:
        L, H, D, B = 32, 32, 128, 16
        S = 32 if num_seqs is None else num_seqs
        lens = r.integers(256, 2048, size=32, endpoint=True)[:S]
        lens = np.maximum(1, np.round(lens * len_scale)).astype(np.int64)
        B = block_size or B
        steps = 8 if decode_steps is None else decode_steps
        need = sum(_ceil_div(int(t) + steps, B) for t in lens)
        N = int(math.ceil(1.3 * need))
        script = [("admit", s, int(t)) for s, t in enumerate(lens)]
        return _finish(2, "7b", num_layers or L, H, D, B, lens, script, steps, seed, N, layout,
                       "32 layers, 32x128 heads, B=16, batch 32, lens U[256,2048], pool 1.3x")
    if index == 3:
        L, H, D, B = 32, 32, 128, 16
        S = 64 if num_seqs is None else num_seqs
        prefix = max(1, int(round(520 * len_scale)))
        suffix = r.integers(64, 512, size=64, endpoint=True)[:S]
        suffix = np.maximum(1, np.round(suffix * len_scale)).astype(np.int64)
        B = block_size or B
        steps = 64 if decode_steps is None else decode_steps
        if prefix_mode == "fork":
            script = [("admit", 0, prefix)] + [("fork", 0, s) for s in range(1, S)]
            script.append(("write", [int(x) for x in suffix]))
        elif prefix_mode == "hash":
            tr = _rng(seed, 5)
            shared = [int(t) for t in tr.integers(0, 32000, size=prefix)]
            script = [("prompt", s, shared + [int(t) for t in tr.integers(0, 32000, size=int(suffix[s]))])
                      for s in range(S)]
        else:
            raise ValueError(prefix_mode)
        lens = prefix + suffix
        shared = _ceil_div(prefix, B)
        need = shared + S + sum(_ceil_div(int(t) + steps, B) - shared for t in lens)
        N = int(math.ceil(1.3 * need))
        return _finish(3, "prefix" if prefix_mode == "fork" else "prefix-hash", num_layers or L, H, D, B, lens,
                       script, steps, seed, N, layout,
                       "7B shape, B=16, 64 seqs share a 520-token prefix, suffix U[64,512], "
                       + ("COW" if prefix_mode == "fork" else "found by block hash"))
    if index == 4:
        L, H, D, B = 40, 40, 128, 32
        S = 128 if num_seqs is None else num_seqs
        sigma = math.sqrt(2.0 * math.log(512.0 / 300.0))
        lens = np.clip(np.round(r.lognormal(math.log(300.0), sigma, size=128)), 16, 4096)[:S]
        lens = np.maximum(1, np.round(lens * len_scale)).astype(np.int64)
        B = block_size or B
        steps = 8 if decode_steps is None else decode_steps
        need = [_ceil_div(int(t) + steps, B) for t in lens]
        N = int(math.ceil(sum(need) / 0.6))
        script = _churn_script(_rng(seed, 3), [int(t) for t in lens], B, N, 0.9)
        return _finish(4, "13b", num_layers or L, H, D, B, lens, script, steps, seed, N, layout,
                       "40 layers, 40x128 heads, B=32, batch 128, lognormal lens, pool 90% after churn")
    if index == 5:
        L, H, D, B = 32, 32, 128, 256
        S = 16 if num_seqs is None else num_seqs
        lens = r.integers(4096, 16384, size=16, endpoint=True)[:S]
        lens = np.maximum(1, np.round(lens * len_scale)).astype(np.int64)
        B = block_size or B
        steps = 4 if decode_steps is None else decode_steps
        need = sum(_ceil_div(int(t) + steps, B) for t in lens)
        N = int(math.ceil(1.3 * need))
        script = [("admit", s, int(t)) for s, t in enumerate(lens)]
        return _finish(5, "long", num_layers or L, H, D, B, lens, script, steps, seed, N, layout,
                       f"32x128 heads, B={B}, batch 16, lens U[4096,16384], shuffled pages")
    raise ValueError(f"unknown workload {index}")


def _churn_script(rng: np.random.Generator, lens: List[int], block_size: int, N: int, fill: float) -> list:
    """Admissions of the batch interleaved with dummy alloc/free until ``fill`` x N blocks are held.

    The block counts here only keep the random draw inside the pool (the batch
    always fits, the final occupancy is ``fill``); the allocator is not modelled.
    """
    target = int(fill * N)
    init = [-(-t // block_size) for t in lens]
    held = 0
    dummies: dict = {}
    next_dummy = 0
    ops: list = []
    s = 0
    S = len(lens)
    while s < S or held < target:
        u = rng.random()
        room = target - held - sum(init[s:])
        if s < S and u < 0.25:
            ops.append(("admit", s, lens[s]))
            held += init[s]
            s += 1
        elif u < 0.7 and room > 0:
            n = min(int(rng.integers(1, 33)), room)
            ops.append(("dummy_alloc", next_dummy, n))
            dummies[next_dummy] = n
            held += n
            next_dummy += 1
        elif dummies:
            keys = sorted(dummies)
            d = keys[int(rng.integers(0, len(keys)))]
            ops.append(("dummy_free", d))
            held -= dummies.pop(d)
    return ops


# --------------------------------------------------------------------------------
# values
# --------------------------------------------------------------------------------

def normal_fp16(seed: int, tag: Tuple[int, ...], shape: Sequence[int]) -> np.ndarray:
    """fp16 draws of N(0, 1) (NumPy; bit-reproducible on any host)."""
    g = _rng(seed, *tag)
    return g.standard_normal(size=tuple(shape), dtype=np.float32).astype(np.float16)


def pool_shape(w: Workload) -> Tuple[int, ...]:
    """Shape of one of the K / V pools, all layers: [L, N, <block>, D]."""
    if w.layout == "NHD":
        return (w.num_layers, w.num_blocks, w.block_size, w.num_heads, w.head_dim)
    return (w.num_layers, w.num_blocks, w.num_heads, w.block_size, w.head_dim)


def pool_scale_shape(w: Workload) -> Tuple[int, ...]:
    """Shape of a per-(token, head) scale pool (E4M3 cache): [L, N, H, B]."""
    return (w.num_layers, w.num_blocks, w.num_heads, w.block_size)


def pool_codes_e4m3(w: Workload, which: int) -> np.ndarray:
    """Initial E4M3 codes of the K (0) / V (1) pool: uniform over the 254 finite codes."""
    g = _rng(w.seed, 110 + which)
    c = g.integers(0, 126, size=pool_shape(w), dtype=np.int64)          # 0x00..0x7D
    c = c + (c >= 0x7F)                                                   # never 0x7F (NaN)
    sign = g.integers(0, 2, size=pool_shape(w), dtype=np.int64) << 7
    return (c | sign).astype(np.uint8)


def pool_scales(w: Workload, which: int) -> np.ndarray:
    """Initial per-(token, head) scales of the K (0) / V (1) pool: U[0.001, 0.01]."""
    return _rng(w.seed, 120 + which).uniform(0.001, 0.01, size=pool_scale_shape(w)).astype(np.float32)


def pool_values(w: Workload, which: int) -> np.ndarray:
    """Initial contents of the K (which=0) or V (which=1) pool: every slot is a draw."""
    return normal_fp16(w.seed, (100 + which,), pool_shape(w))


def query_values(w: Workload, step: int, layer: int) -> np.ndarray:
    return normal_fp16(w.seed, (200, step, layer), (w.num_seqs, w.num_heads, w.head_dim))


def new_token_values(w: Workload, step: int, layer: int, which: int) -> np.ndarray:
    """K (which=0) / V (which=1) of the token each sequence appends at ``step``."""
    return normal_fp16(w.seed, (300 + which, step, layer), (w.num_seqs, w.num_heads, w.head_dim))


def write_values(w: Workload, op_index: int, layer: int, which: int, num_tokens: int) -> np.ndarray:
    """K / V of the tokens a ``("write", counts)`` op appends, in (sequence, token) order."""
    return normal_fp16(w.seed, (400 + which, op_index, layer), (num_tokens, w.num_heads, w.head_dim))


def torch_normal_fp16(seed: int, tag: Tuple[int, ...], shape: Sequence[int], device):
    """fp16 draws of N(0, 1) made on ``device`` by torch (used for pools too big for the host)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([int(seed)] + [int(t) for t in tag]).generate_state(1)[0]))
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float16)


def torch_e4m3_pool(w: Workload, which: int, device):
    """E4M3 codes and scales of a pool made on ``device`` by torch (pools too big for the host)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([int(w.seed), 110 + which]).generate_state(1)[0]))
    c = torch.randint(0, 126, pool_shape(w), generator=g, device=device, dtype=torch.int16)
    c = c + (c >= 0x7F).to(torch.int16)
    c = c | (torch.randint(0, 2, pool_shape(w), generator=g, device=device, dtype=torch.int16) << 7)
    s = torch.rand(pool_scale_shape(w), generator=g, device=device, dtype=torch.float32) * 0.009 + 0.001
    return c.to(torch.uint8), s
