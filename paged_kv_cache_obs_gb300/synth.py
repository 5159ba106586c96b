"""Seeded synthetic workloads for the compression pass and the decode consumer.

This module only draws inputs: KV pools, block tables, window queries and carried global
scores with the shapes and value distributions of the five workloads.  It holds none of the
method's arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Workloads (sizes as in the workload list of this project):
  tiny         1 request, 1 layer, H_q 4 / H_kv 2, d 64, b 16, N_max 8, w 8; K,V,Q ~ N(0,1); G = 0
  qwen2_7b     28 layers, 28 / 4 heads, d 128, b 32, N_max 64, w 16, 32 requests; K,V ~ N(0,1) with
               rotate-half RoPE (theta 1e6) on K at positions 0..L-1 and on the window queries at
               L-w+i; G ~ U(0,1)
  llama3_8b    32 layers, 32 / 8 heads, d 128, b 16, N_max 128, w 32, 64 requests; keys = one of
               two per-block centroids (64 centroids ~ N(0,1) per layer and head) + 0.05*N(0,1),
               10% of positions per head are heavy hitters scaled x4; V, Q ~ N(0,1); G ~ U(0,1)
  shared_prefix llama3_8b shape with N_max 96, 64 requests whose first 16 blocks are the same
               physical blocks (refcount 64 requests + 1 prefix-cache reference)
  mixed        llama3_8b shape, 256 running requests: 32 hold query slots at N_max = 128 full
               blocks and compress; 224 decode with U{1..128} blocks and a last-block fill of
               U{1..16} tokens
  prefill      llama3_8b shape with N_max 64 (k = 1008): 64 requests that left a long prefill and
               hold U{1009..2048} tokens each (first compression after the prompt); G ~ U(0,1)
  prefill_long llama3_8b shape with N_max 128 (k = 2032): 16 requests holding U{2033..8192}
               tokens each (prompts beyond one cluster: the multi-pass form)
Physical block ids are a seeded random permutation over the pool in every workload.
Seeds: 0x5A1F0000 + workload index.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    index: int
    num_requests: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    n_max: int
    window: int
    key_recipe: str = "normal"        # normal | rope | clustered
    global_init: str = "uniform"      # zeros | uniform
    shared_prefix_blocks: int = 0
    num_decode: int = 0               # mixed workload: requests that only decode
    prefill_max: int = 0              # > n_max*b: compressing requests hold U{k+1..prefill_max} tokens
    budget_min: int = 0               # > 0: per-request budgets N_max_r ~ U{budget_min..n_max}, each
                                      # request at its own trigger (N_max_r full blocks)
    pool_blocks: int = 0              # 0 = just enough (+ targets), else this many
    alpha: float = 0.5
    beta: float = 0.5
    decay: float = 0.9
    protect_window: int = 1
    causal: int = 1
    rope_theta: float = 1e6

    @property
    def L(self) -> int:
        return self.n_max * self.block_size

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def params(self) -> dict:
        return dict(num_layers=self.num_layers, num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    block_size=self.block_size, n_max=self.n_max, window=self.window,
                    alpha=self.alpha, beta=self.beta, decay=self.decay, scale=self.scale,
                    protect_window=self.protect_window, causal=self.causal)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 1, 4, 2, 64, 16, 8, 8, global_init="zeros"),
    "qwen2_7b": Workload("qwen2_7b", 1, 32, 28, 28, 4, 128, 32, 64, 16, key_recipe="rope"),
    "llama3_8b": Workload("llama3_8b", 2, 64, 32, 32, 8, 128, 16, 128, 32, key_recipe="clustered"),
    "shared_prefix": Workload("shared_prefix", 3, 64, 32, 32, 8, 128, 16, 96, 32,
                              key_recipe="clustered", shared_prefix_blocks=16),
    "mixed": Workload("mixed", 4, 32, 32, 32, 8, 128, 16, 128, 32, key_recipe="clustered",
                      num_decode=224),
    "prefill": Workload("prefill", 5, 64, 32, 32, 8, 128, 16, 64, 32, key_recipe="clustered",
                        prefill_max=2048),
    # prompts beyond one cluster (up to 8192 tokens): the multi-pass form of the pass
    "prefill_long": Workload("prefill_long", 6, 16, 32, 32, 8, 128, 16, 128, 32, key_recipe="clustered",
                             prefill_max=8192),
}


def seed_of(wl: Workload) -> int:
    return 0x5A1F0000 + wl.index


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _rope_(x: torch.Tensor, pos: torch.Tensor, theta: float):
    """Rotate-half rotary embedding applied in fp32 to x[..., d] at integer positions pos[...]."""
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-torch.arange(0, half, device=x.device, dtype=torch.float64) * 2.0 / d)
    ang = pos.to(torch.float64)[..., None] * inv
    cos, sin = ang.cos().to(torch.float32), ang.sin().to(torch.float32)
    x1, x2 = x[..., :half].clone(), x[..., half:].clone()
    x[..., :half] = x1 * cos - x2 * sin
    x[..., half:] = x2 * cos + x1 * sin
    return x


@dataclasses.dataclass
class Inputs:
    wl: Workload
    pool: torch.Tensor             # bf16 [layers, NB, 2, Hkv, b, d]
    block_tables: np.ndarray       # int32 [R_all, max_blocks] (host)
    seq_len: np.ndarray            # int32 [R_all]
    qslot: np.ndarray              # int32 [R_compress] (compressing requests are rows 0..R-1)
    obs_q: torch.Tensor            # bf16 [M, layers, w, Hq, d]
    global_scores: torch.Tensor    # fp32 [M, layers, Hkv, L]
    refcount: np.ndarray           # int32 [NB] refcount of every physical block
    num_compress: int
    decode_q: torch.Tensor | None  # bf16 [layers, num_decode, Hq, d] (mixed workload)
    n_max_req: np.ndarray | None = None  # int32 [R] per-request budgets (or None)


def make_inputs(wl: Workload, device="cpu", seed: int | None = None) -> Inputs:
    """Draw one workload.  Compressing requests are rows 0..R-1 of the tables, decode-only
    requests (mixed workload) follow.  Query slot of compressing request r is r."""
    seed = seed_of(wl) if seed is None else seed
    dev = torch.device(device)
    g = _gen(dev, seed)
    rng = np.random.default_rng(seed)
    R, nl, Hq, Hkv, d, b, n_max, w = (wl.num_requests, wl.num_layers, wl.num_q_heads,
                                      wl.num_kv_heads, wl.head_dim, wl.block_size, wl.n_max,
                                      wl.window)
    L = wl.L
    P = wl.shared_prefix_blocks

    # ---- logical -> physical block assignment ---------------------------------------
    counts = [n_max] * R
    fills = [b] * R
    L_row = L  # row length of the global scores: the longest sequence
    if wl.prefill_max > L:
        k_keep = (n_max - 1) * b
        lens = rng.integers(k_keep + 1, wl.prefill_max + 1, size=R)
        counts = [int((x + b - 1) // b) for x in lens]
        fills = [int(x - (c - 1) * b) for x, c in zip(lens, counts)]
        L_row = wl.prefill_max
    n_max_req = None
    if wl.budget_min:
        n_max_req = rng.integers(wl.budget_min, n_max + 1, size=R).astype(np.int32)
        counts = [int(x) for x in n_max_req]
    if wl.num_decode:
        counts += list(rng.integers(1, n_max + 1, size=wl.num_decode))
        fills += list(rng.integers(1, b + 1, size=wl.num_decode))
    R_all = len(counts)
    needed = P + sum(c - (P if i < R else 0) for i, c in enumerate(counts))
    targets = R * P  # fresh blocks the shared-prefix plan will need
    NB = wl.pool_blocks or int(needed + targets + max(16, needed // 64))
    assert NB >= needed + targets
    perm = rng.permutation(NB).astype(np.int32)
    max_blocks = max(n_max, max(counts), (L_row + b - 1) // b)
    tables = np.full((R_all, max_blocks), -1, dtype=np.int32)
    nxt = 0
    shared = perm[nxt:nxt + P]
    nxt += P
    refcount = np.zeros(NB, dtype=np.int32)
    refcount[shared] = R + 1 if P else 0  # every request + the prefix cache's own reference
    for r, c in enumerate(counts):
        start = 0
        if r < R and P:
            tables[r, :P] = shared
            start = P
        tables[r, start:c] = perm[nxt:nxt + c - start]
        refcount[perm[nxt:nxt + c - start]] = 1
        nxt += c - start
    seq_len = np.array([(c - 1) * b + f for c, f in zip(counts, fills)], dtype=np.int32)

    # ---- logical position of every physical row (for RoPE and per-block recipes) ------
    phys_pos = torch.full((NB,), -1, dtype=torch.int64)
    for r, c in enumerate(counts):
        for i in range(c):
            phys_pos[int(tables[r, i])] = i  # logical block index (shared blocks: same index)
    phys_pos = phys_pos.to(dev)

    # ---- KV pool, one layer at a time ---------------------------------------------------
    # A requested pool far larger than the blocks in use (the mixed workload's 120k blocks) is left
    # uninitialised except for the referenced blocks: the kernels read only blocks of some
    # table (a target block is written before it is read).  Otherwise every block is drawn.
    sparse = bool(wl.pool_blocks) and NB > 4 * (needed + targets)
    if sparse:
        pool = torch.empty((nl, NB, 2, Hkv, b, d), dtype=torch.bfloat16, device=dev)
        ids = torch.as_tensor(np.nonzero(refcount)[0], dtype=torch.int64, device=dev)
    else:
        pool = torch.zeros((nl, NB, 2, Hkv, b, d), dtype=torch.bfloat16, device=dev)
        ids = None
    nfill = NB if ids is None else int(ids.numel())
    fpos = phys_pos if ids is None else phys_pos[ids]
    for l in range(nl):
        if wl.key_recipe == "clustered":
            cent = torch.randn((Hkv, 64, d), generator=g, device=dev)
            pick = torch.randint(0, 64, (nfill, Hkv, 2), generator=g, device=dev)
            which = torch.randint(0, 2, (nfill, Hkv, b), generator=g, device=dev)
            cid = torch.gather(pick, 2, which)  # [blocks, Hkv, b] centroid of each token
            hidx = torch.arange(Hkv, device=dev)[None, :, None].expand_as(cid)
            k = cent[hidx, cid] + 0.05 * torch.randn((nfill, Hkv, b, d), generator=g, device=dev)
            heavy = torch.rand((nfill, Hkv, b), generator=g, device=dev) < 0.10
            k = torch.where(heavy[..., None], 4.0 * k, k)
        else:
            k = torch.randn((nfill, Hkv, b, d), generator=g, device=dev)
            if wl.key_recipe == "rope":
                pos = fpos.clamp(min=0)[:, None, None] * b + torch.arange(b, device=dev)[None, None, :]
                k = _rope_(k, pos.expand(nfill, Hkv, b), wl.rope_theta)
        v = torch.randn((nfill, Hkv, b, d), generator=g, device=dev)
        if ids is None:
            pool[l, :, 0] = k.to(torch.bfloat16)
            pool[l, :, 1] = v.to(torch.bfloat16)
        else:
            pool[l].index_copy_(0, ids, torch.stack((k, v), dim=1).to(torch.bfloat16))
        del k, v

    # ---- window queries and carried global scores (one query slot per compressing request)
    M = R
    q = torch.randn((M, nl, w, Hq, d), generator=g, device=dev)
    if wl.key_recipe == "rope":
        last = torch.as_tensor(seq_len[:M], device=dev, dtype=torch.int64)
        pos = (last[:, None] - w + torch.arange(w, device=dev)[None, :])[:, None, :, None].expand(M, nl, w, Hq)
        q = _rope_(q, pos, wl.rope_theta)
    obs_q = q.to(torch.bfloat16)
    if wl.global_init == "zeros":
        gs = torch.zeros((M, nl, Hkv, L_row), dtype=torch.float32, device=dev)
    else:
        gs = torch.rand((M, nl, Hkv, L_row), generator=g, device=dev, dtype=torch.float32)

    decode_q = None
    if wl.num_decode:
        decode_q = torch.randn((nl, wl.num_decode, Hq, d), generator=g, device=dev).to(torch.bfloat16)

    return Inputs(wl=wl, pool=pool, block_tables=tables, seq_len=seq_len,
                  qslot=np.arange(R, dtype=np.int32), obs_q=obs_q, global_scores=gs,
                  refcount=refcount, num_compress=R, decode_q=decode_q, n_max_req=n_max_req)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
