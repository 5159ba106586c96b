"""Plain CPU oracle for the Compressed-PagedAttention compression pass of Zipage.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, by the smoke check in
``__graft_entry__.py`` and by the CPU-baseline leg of ``bench.py``; the product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

Everything here is deliberately slow and literal: fp64 arithmetic from the exact bf16 input
values, one (request, layer, kv-head) unit at a time, no blocking, no fusion.  A library
matmul or sort stands for one step where the definition is a matmul or a sort.

Sources (the pages are four summaries of the paper "Zipage: Maintain High Request Concurrency
for LLM Reasoning through Compressed PagedAttention", arXiv 2603.08743, on gist.science):

* zh page, section 2.1 ("核心机制：压缩 PagedAttention"): the per-request cap of N_max blocks of b
  tokens, the trigger, the observation window of the last w queries, the three scores
  (attention, redundancy, global from historical attention), keeping k = (N_max-1)*b tokens
  compacted into the first N_max-1 blocks and freeing the rest, the O(N*b^2) Lightning
  Redundancy Score that only looks inside a block.
* zh page, section 2.2 ("混合调度策略"), de page section 2 ("Prefix Caching für komprimierte
  Daten"), fr page section 2.C: shared prefix blocks (refcount > 1) are not moved; the
  compressed data goes to newly allocated target blocks.
* fr page, section 2.A: the last w tokens (the observation window) are always kept.
* de page, section 2 ("Lightning Redundancy Score"): the redundancy is computed block by
  block without materialising the full similarity matrix.

Readings where the pages are silent:

* scale = 1/sqrt(d) (the usual attention scale);
* the observation-window query i is the query of token position L-w+i and attends causally,
  i.e. to keys t <= L-w+i;
* GQA grouping is contiguous: kv head h serves query heads h*G .. h*G+G-1;
* attention score of token t = mean over the w*G window rows of the row softmax;
* redundancy of t = mean cosine similarity of k_t to the other keys of its own block
  (cosine with norms clamped at 1e-12; a block of one token has redundancy 0);
* S = attn + alpha*G - beta*R with the carried global score G from *before* this pass;
* protected window: S = +inf for the last w tokens when protect_window is set;
* keep the k tokens first in the order (S descending, position ascending), i.e. on equal S
  the earlier token is kept; NaN ranks as -inf;
* global update G'[j] = decay*G[src_j] + attn[src_j] for the k survivors, 0 for j >= k;
* target blocks replace exactly the leading blocks whose refcount is > 1, lowest free id
  first; the old last block is released (decref), replaced shared blocks are decref'd.
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------------------
# bf16 <-> float helpers.  bf16 values travel as their 16-bit patterns (uint16 arrays) so
# that "bit-exact" comparisons of compacted K/V are comparisons of integers.
# ----------------------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of each bf16 bit pattern, as float64 (bf16 is the top half of a float32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 (via float32, then round-to-nearest-even on the low 16 bits)."""
    f32 = np.asarray(x, dtype=np.float32)
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(f32)
    out = rounded.astype(np.uint16)
    out[nan] = np.uint16(0x7FC0)
    return out


# ----------------------------------------------------------------------------------------
# Step 1 — observation-window attention score (zh 2.1 "观察窗口"/"评分机制"; de 2
# "Observation Window"; es 2 "ventana de observación").
# ----------------------------------------------------------------------------------------


def window_attention(q: np.ndarray, k: np.ndarray, scale: float, causal: bool = True) -> np.ndarray:
    """Attention that the observation window pays to each cached token.

    q: [w, G, d] float64, the window queries of the G query heads of one kv head; row i is the
       query of token position L-w+i.
    k: [L, d] float64, all cached keys of that kv head in logical order.
    Returns attn[L] = (1/(w*G)) * sum_{i,g} softmax_t(scale * <q[i,g], k_t>) over the keys the
    row may see (t <= L-w+i when causal).
    """
    w, G, _ = q.shape
    L = k.shape[0]
    attn = np.zeros(L, dtype=np.float64)
    for i in range(w):
        visible = L - w + i + 1 if causal else L
        for g in range(G):
            z = scale * (k[:visible] @ q[i, g])  # logits of this window row
            z = z - z.max()
            p = np.exp(z)
            p /= p.sum()
            attn[:visible] += p
    return attn / (w * G)


# ----------------------------------------------------------------------------------------
# Step 2 — Lightning Redundancy Score (zh 2.1 "闪电冗余分数"; de 2 "Lightning Redundancy
# Score"; es 2 "Optimizaciones de Kernel"; fr 2.E).  Only pairs inside one block of b tokens
# are compared: N blocks x b^2 pairs instead of (N*b)^2.
# ----------------------------------------------------------------------------------------


def lightning_redundancy(k: np.ndarray, b: int) -> np.ndarray:
    """R[t] = mean over the other tokens j of t's block of cos(k_t, k_j); 0 for a lone token."""
    L = k.shape[0]
    R = np.zeros(L, dtype=np.float64)
    for start in range(0, L, b):
        blk = k[start:start + b]
        m = blk.shape[0]
        if m < 2:
            continue
        norms = np.maximum(np.sqrt((blk * blk).sum(axis=1)), 1e-12)
        unit = blk / norms[:, None]
        gram = unit @ unit.T  # b x b cosine matrix of this block only
        R[start:start + m] = (gram.sum(axis=1) - np.diag(gram)) / (m - 1)
    return R


def all_pairs_redundancy(k: np.ndarray) -> np.ndarray:
    """The original redundancy that Lightning replaces (zh 2.1, es 2: O(N^2 b^2) pairs over the
    N blocks of b tokens; de 2: it needs the full similarity matrix): R[t] = mean over every
    other token j of the sequence of cos(k_t, k_j).  Same cosine and clamp as the Lightning
    form; a sequence of one token has redundancy 0.  The full L x L cosine matrix is formed,
    as that method does."""
    L = k.shape[0]
    R = np.zeros(L, dtype=np.float64)
    if L < 2:
        return R
    norms = np.maximum(np.sqrt((k * k).sum(axis=1)), 1e-12)
    unit = k / norms[:, None]
    cos = unit @ unit.T  # L x L
    return (cos.sum(axis=1) - np.diag(cos)) / (L - 1)


# ----------------------------------------------------------------------------------------
# Step 3 — combined importance score (zh 2.1 "评分机制": attention + redundancy + global).
# ----------------------------------------------------------------------------------------


def combine_scores(attn, G, R, alpha: float, beta: float, window: int, protect_window: bool):
    """S = attn + alpha*G - beta*R; the last `window` tokens get +inf when protected (fr 2.A)."""
    S = np.asarray(attn, np.float64) + alpha * np.asarray(G, np.float64) - beta * np.asarray(R, np.float64)
    if protect_window and window > 0:
        S = S.copy()
        S[-window:] = np.inf
    return S


# ----------------------------------------------------------------------------------------
# Step 4 — per-head top-k retention (zh 2.1 "保留策略": keep the k = (N_max-1)*b highest).
# ----------------------------------------------------------------------------------------


def select_keep(S: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k kept tokens, in ascending (original) order.

    Ranking: higher S first; on equal S the earlier position first; NaN ranks last.
    """
    L = len(S)
    if k >= L:
        return np.arange(L, dtype=np.int64)

    def rank_key(t):
        s = float(S[t])
        if math.isnan(s):
            s = -math.inf
        return (-s, t)

    order = sorted(range(L), key=rank_key)
    return np.array(sorted(order[:k]), dtype=np.int64)


# ----------------------------------------------------------------------------------------
# Step 5 — global score carried across compressions (zh 2.1 "全局分数，来自历史注意力";
# zh 2.3 "全局分数更新"; fr 2.E "Score Global").
# ----------------------------------------------------------------------------------------


def global_update(G, attn, src: np.ndarray, decay: float, L: int) -> np.ndarray:
    """G'[j] = decay*G[src_j] + attn[src_j] for j < k, and 0 for k <= j < L."""
    out = np.zeros(L, dtype=np.float64)
    out[:len(src)] = decay * np.asarray(G, np.float64)[src] + np.asarray(attn, np.float64)[src]
    return out


# ----------------------------------------------------------------------------------------
# Step 6 — physical placement: target blocks for shared prefix blocks (zh 2.2 "前缀缓存兼容";
# de 2 "Prefix Caching"; fr 2.C) and release of the last block (zh 2.1 "释放剩余块").
# ----------------------------------------------------------------------------------------


def plan_dst_table(table, n_max: int, refcount: dict, free_ids: list):
    """Destination table for one request.

    Logical blocks i < n_max-1 keep their physical id unless it is shared (refcount > 1); a
    shared block is replaced by a fresh block, taken lowest free id first.  `free_ids` is a
    sorted list and is consumed.  Returns (dst_table[n_max-1], replaced_ids).
    """
    dst, replaced = [], []
    for i in range(n_max - 1):
        blk = int(table[i])
        if refcount.get(blk, 0) > 1:
            dst.append(free_ids.pop(0))
            replaced.append(blk)
        else:
            dst.append(blk)
    return dst, replaced


def slot_location(table, slot: int, b: int):
    """Logical slot -> (physical block id, row inside the block)."""
    return int(table[slot // b]), slot % b


# ----------------------------------------------------------------------------------------
# One unit (request, layer, kv head) and the whole pass.
# ----------------------------------------------------------------------------------------


def score_unit(q_bits, k_bits, G, *, b, n_max, window, alpha, beta, scale, protect_window, causal):
    """Scores of one unit.  q_bits [w, G, d] and k_bits [L, d] are bf16 patterns, G [L] float."""
    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    attn = window_attention(q, k, scale, causal)
    R = lightning_redundancy(k, b)
    S = combine_scores(attn, G, R, alpha, beta, window, protect_window)
    return attn, R, S


def compress_pass(pool, block_tables, dst_tables, seq_len, qslot, obs_q, global_scores, p,
                  units=None, n_max_per_req=None):
    """The compression pass over every (request, layer, kv head) unit, on copies of the state.

    pool          uint16 [layers, num_blocks, 2, Hkv, b, d]   (index 0 = K, 1 = V)
    block_tables  int32  [R, max_blocks]   physical ids of the logical blocks (source)
    dst_tables    int32  [R, max_blocks]   physical ids the survivors are written to
    seq_len       int32  [R]               cached tokens (= n_max*b at the trigger)
    qslot         int32  [R]               query slot of each request
    obs_q         uint16 [M, layers, w, Hq, d]
    global_scores float32 [M, layers, Hkv, n_max*b]
    p             dict with num_q_heads, num_kv_heads, block_size, n_max, window, alpha, beta,
                  decay, scale, protect_window, causal
    units         optional iterable of (r, layer, h) to compute; default all.
    n_max_per_req optional per-request block budgets (default p["n_max"] for every request);
                  request r keeps k_r = (N_max_r - 1) * b tokens per head.

    Returns (new_pool, new_global_scores, debug) where debug maps (r, layer, h) to a dict with
    attn, R, S (float64 [L]) and src (int64 [k]).  Units are independent: every read of the
    pass happens on the input copy, every write on the output copy.
    """
    layers, _, _, Hkv, b, d = pool.shape
    Hq = p["num_q_heads"]
    Gq = Hq // Hkv
    w = p["window"]
    new_pool = pool.copy()
    new_G = np.array(global_scores, dtype=np.float32, copy=True)
    debug = {}
    R_req = block_tables.shape[0]
    if units is None:
        units = [(r, l, h) for r in range(R_req) for l in range(layers) for h in range(Hkv)]
    for (r, l, h) in units:
        L = int(seq_len[r])
        n_max = int(n_max_per_req[r]) if n_max_per_req is not None else p["n_max"]
        k_keep = (n_max - 1) * b
        table, dtab = block_tables[r], dst_tables[r]
        rows = [slot_location(table, t, b) for t in range(L)]
        k_bits = np.stack([pool[l, blk, 0, h, row] for blk, row in rows])
        v_bits = np.stack([pool[l, blk, 1, h, row] for blk, row in rows])
        s = int(qslot[r])
        q_bits = obs_q[s, l, :, h * Gq:(h + 1) * Gq, :]
        G = global_scores[s, l, h, :L].astype(np.float64)
        attn, R, S = score_unit(q_bits, k_bits, G, b=b, n_max=n_max, window=w,
                                alpha=p["alpha"], beta=p["beta"], scale=p["scale"],
                                protect_window=p["protect_window"], causal=p["causal"])
        src = select_keep(S, k_keep)
        for j, t in enumerate(src):
            blk, row = slot_location(dtab, j, b)
            new_pool[l, blk, 0, h, row] = k_bits[t]
            new_pool[l, blk, 1, h, row] = v_bits[t]
        new_G[s, l, h, :L] = global_update(G, attn, src, p["decay"], L)
        debug[(r, l, h)] = {"attn": attn, "R": R, "S": S, "src": src}
    return new_pool, new_G, debug


def compact_unit_with(src, k_bits, v_bits):
    """Compacted (K, V) rows of one unit for a given survivor list: row j is input row src[j]."""
    src = np.asarray(src, dtype=np.int64)
    return k_bits[src], v_bits[src]


# ----------------------------------------------------------------------------------------
# Consumer — paged decode attention over the compacted cache (zh 2.3 "支持 ... FlashAttention";
# the decode side of the asynchronous compression in zh 2.1 / fr 2.D).
# ----------------------------------------------------------------------------------------


def decode_attention(q_bits, k_bits, v_bits, scale: float) -> np.ndarray:
    """One new token per request: out[g] = softmax(scale*q_g.K^T) V, fp64.

    q_bits [G, d], k_bits [n, d], v_bits [n, d] (bf16 patterns) -> out [G, d] float64.
    """
    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    v = bf16_bits_to_f64(v_bits)
    out = np.zeros((q.shape[0], v.shape[1]), dtype=np.float64)
    for g in range(q.shape[0]):
        z = scale * (k @ q[g])
        z = z - z.max()
        pr = np.exp(z)
        pr /= pr.sum()
        out[g] = pr @ v
    return out


def gather_rows(pool, layer, kv, h, table, n, b):
    """Logical rows 0..n-1 of one (layer, K|V, head) through a block table."""
    return np.stack([pool[layer, int(table[t // b]), kv, h, t % b] for t in range(n)])


# ----------------------------------------------------------------------------------------
# Block pool with reference counts (the PagedAttention block manager the pages build on:
# zh 2.2 prefix sharing; fr 2.C "blocs partagés").  A literal model used to check the
# library's allocator: lowest free id first, all-or-nothing allocation.
# ----------------------------------------------------------------------------------------


class RefcountPool:
    def __init__(self, num_blocks: int):
        self.refcount = [0] * num_blocks

    def free_ids(self):
        return [i for i, c in enumerate(self.refcount) if c == 0]

    def alloc(self, n: int):
        free = self.free_ids()
        if len(free) < n:
            return None
        ids = free[:n]
        for i in ids:
            self.refcount[i] = 1
        return ids

    def incref(self, ids):
        for i in ids:
            self.refcount[int(i)] += 1

    def decref(self, ids):
        for i in ids:
            self.refcount[int(i)] -= 1

    def num_free(self):
        return len(self.free_ids())
