"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one step of the compression pass (Zipage summaries on gist.science: zh page
section 2.1, de page section 2, fr page section 2.A/2.C/2.E) against a hand-worked example, a
closed form, a special case with a known answer, an invariant, or an independent brute-force
formulation on a tiny input.  A dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import zipage_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _two_block():
    with open(os.path.join(GOLDEN, "two_block_example.json")) as f:
        ex = json.load(f)
    q = np.array([[[math.sqrt(2.0), 0.0]]])  # [w=1, G=1, d=2]
    k = np.array([[0.0, 1.0], [math.log(2), 0.0], [math.log(3), 0.0], [math.log(4), 0.0]])
    return ex, q, k


# ---------------------------------------------------------------- window attention --------

def test_two_block_hand_example_attention():
    ex, q, k = _two_block()
    attn = O.window_attention(q, k, scale=1 / math.sqrt(2), causal=True)
    np.testing.assert_allclose(attn, ex["attn"], rtol=0, atol=1e-15)


def test_two_block_hand_example_redundancy():
    ex, q, k = _two_block()
    np.testing.assert_allclose(O.lightning_redundancy(k, 2), ex["redundancy"], atol=1e-15)


@pytest.mark.parametrize("case", range(5))
def test_two_block_hand_example_scores_and_selection(case):
    ex, q, k = _two_block()
    c = ex["cases"][case]
    attn = O.window_attention(q, k, 1 / math.sqrt(2), True)
    R = O.lightning_redundancy(k, 2)
    S = O.combine_scores(attn, np.array(c["G"], float), R, c["alpha"], c["beta"], ex["w"],
                         bool(c["protect_window"]))
    want = [math.inf if s == "inf" else s for s in c["S"]]
    np.testing.assert_allclose(S, want, atol=1e-15)
    assert list(O.select_keep(S, ex["k"])) == c["keep"]


@pytest.mark.parametrize("case", range(5))
def test_two_block_hand_example_global_update(case):
    # The carried global score after the pass (zh 2.1 "global score from historical attention",
    # fr 2.E), worked by hand in the golden file from the hand-derived attention and keep set:
    # survivor j carries decay*G + attn of its source token, the freed slots hold 0.
    ex, _, _ = _two_block()
    c = ex["cases"][case]
    got = O.global_update(np.array(c["G"], float), np.array(ex["attn"], float), np.array(c["keep"]),
                          ex["decay"], ex["L"])
    np.testing.assert_allclose(got, c["G_new"], rtol=0, atol=1e-15)


def _rand_qk(rng, w, G, L, d):
    return rng.standard_normal((w, G, d)), rng.standard_normal((L, d))


@pytest.mark.parametrize("causal", [True, False])
def test_attention_mass_is_one(causal):
    rng = np.random.default_rng(1)
    q, k = _rand_qk(rng, 5, 3, 40, 8)
    attn = O.window_attention(q, k, 0.3, causal)
    assert abs(attn.sum() - 1.0) < 1e-12
    assert (attn >= 0).all()


def test_identical_keys_causal_closed_form():
    # All keys equal: every visible key gets 1/(number visible) from each row.
    rng = np.random.default_rng(2)
    L, w, G, d = 24, 6, 2, 8
    q = rng.standard_normal((w, G, d))
    k = np.tile(rng.standard_normal(d), (L, 1))
    attn = O.window_attention(q, k, 0.5, causal=True)
    want = np.array([sum(1.0 / (L - w + i + 1) for i in range(w) if t <= L - w + i) / w
                     for t in range(L)])
    np.testing.assert_allclose(attn, want, rtol=1e-13)
    attn_nc = O.window_attention(q, k, 0.5, causal=False)
    np.testing.assert_allclose(attn_nc, np.full(L, 1.0 / L), rtol=1e-13)


def test_window_row_position_and_mask():
    # Row i sees exactly keys 0..L-w+i: a huge logit on key L-1 only reaches the last row.
    L, w, d = 10, 3, 4
    k = np.zeros((L, d))
    k[L - 1, 0] = 1.0
    q = np.zeros((w, 1, d))
    q[:, 0, 0] = 200.0
    attn = O.window_attention(q, k, 1.0, causal=True)
    # rows 0,1 see keys 0..7 / 0..8 with equal logits 0; row 2 puts ~all mass on key 9
    want = np.zeros(L)
    want[:8] += 1 / 8
    want[:9] += 1 / 9
    want[9] += 1.0
    np.testing.assert_allclose(attn, want / 3, atol=1e-12)


def test_gqa_grouping_is_contiguous():
    # H_q 4 / H_kv 2: kv head 1 is served by query heads 2 and 3 (contiguous grouping).
    from paged_kv_cache_obs_gb300 import synth
    wl = synth.WORKLOADS["tiny"].scaled(n_max=2, window=1, num_q_heads=4, num_kv_heads=2,
                                        protect_window=0, alpha=0.0, beta=0.0)
    b, d, L = wl.block_size, wl.head_dim, wl.L
    pool = np.zeros((1, 2, 2, 2, b, d), dtype=np.uint16)
    one = O.f64_to_bf16_bits(np.array([1.0]))[0]
    # key 5 points along axis 0, key 9 along axis 1, in both kv heads
    for h in range(2):
        pool[0, 0, 0, h, 5, 0] = one
        pool[0, 0, 0, h, 9, 1] = one
    obs_q = np.zeros((1, 1, 1, 4, d), dtype=np.uint16)
    big = O.f64_to_bf16_bits(np.array([64.0]))[0]
    obs_q[0, 0, 0, 0, 1] = big  # query heads 0,1 -> key 9
    obs_q[0, 0, 0, 1, 1] = big
    obs_q[0, 0, 0, 2, 0] = big  # query heads 2,3 -> key 5
    obs_q[0, 0, 0, 3, 0] = big
    tables = np.array([[0, 1]], dtype=np.int32)
    gs = np.zeros((1, 1, 2, L), dtype=np.float32)
    _, _, dbg = O.compress_pass(pool, tables, tables, np.array([L]), np.array([0]), obs_q, gs,
                                wl.params())
    assert int(np.argmax(dbg[(0, 0, 0)]["attn"])) == 9
    assert int(np.argmax(dbg[(0, 0, 1)]["attn"])) == 5


# ---------------------------------------------------------------- redundancy --------------

def _naive_same_block_redundancy(k, b):
    """Independent brute force: full L x L cosine matrix, masked to same-block pairs."""
    L = k.shape[0]
    n = np.maximum(np.linalg.norm(k, axis=1), 1e-12)
    cos = (k @ k.T) / np.outer(n, n)
    R = np.zeros(L)
    for t in range(L):
        same = [j for j in range(L) if j // b == t // b and j != t]
        R[t] = sum(cos[t, j] for j in same) / len(same) if same else 0.0
    return R


@pytest.mark.parametrize("L,b", [(64, 16), (96, 32), (40, 16), (17, 4)])
def test_lightning_equals_all_pairs_same_block(L, b):
    rng = np.random.default_rng(L * 7 + b)
    k = rng.standard_normal((L, 12)) * rng.uniform(0.1, 5, size=(L, 1))
    np.testing.assert_allclose(O.lightning_redundancy(k, b), _naive_same_block_redundancy(k, b),
                               rtol=1e-12, atol=1e-14)


def test_redundancy_special_cases():
    rng = np.random.default_rng(3)
    d, b = 16, 8
    same = np.tile(rng.standard_normal(d), (b, 1)) * rng.uniform(0.5, 2, size=(b, 1))
    np.testing.assert_allclose(O.lightning_redundancy(same, b), np.ones(b), atol=1e-14)
    ortho = np.eye(d)[:b] * 3.0
    np.testing.assert_allclose(O.lightning_redundancy(ortho, b), np.zeros(b), atol=1e-15)
    v = rng.standard_normal(d)
    np.testing.assert_allclose(O.lightning_redundancy(np.stack([v, -2 * v]), 2), [-1, -1],
                               atol=1e-14)
    # a trailing block of one token has redundancy 0
    np.testing.assert_allclose(O.lightning_redundancy(np.ones((3, 4)), 2), [1, 1, 0], atol=1e-14)


def test_all_pairs_redundancy_closed_form():
    """Sum over j != t of cos(k_t, k_j) is unit_t . (sum_j unit_j) - 1, so the all-pairs mean
    needs no matrix: an independent formula for the same quantity."""
    rng = np.random.default_rng(11)
    for L in (2, 5, 64, 257):
        k = rng.standard_normal((L, 24)) * rng.uniform(0.05, 8, size=(L, 1))
        unit = k / np.linalg.norm(k, axis=1, keepdims=True)
        want = (unit @ unit.sum(axis=0) - 1.0) / (L - 1)
        np.testing.assert_allclose(O.all_pairs_redundancy(k), want, rtol=1e-11, atol=1e-13)


def test_all_pairs_redundancy_special_cases():
    rng = np.random.default_rng(12)
    d = 16
    # one block: all pairs are the block's pairs, so it is the Lightning score
    k = rng.standard_normal((16, d))
    np.testing.assert_allclose(O.all_pairs_redundancy(k), O.lightning_redundancy(k, 16), atol=1e-14)
    # identical directions -> 1; orthonormal keys -> 0; a key and its negative -> -1
    same = np.tile(rng.standard_normal(d), (9, 1)) * rng.uniform(0.5, 2, size=(9, 1))
    np.testing.assert_allclose(O.all_pairs_redundancy(same), np.ones(9), atol=1e-14)
    np.testing.assert_allclose(O.all_pairs_redundancy(np.eye(d)[:7] * 2.5), np.zeros(7), atol=1e-15)
    v = rng.standard_normal(d)
    np.testing.assert_allclose(O.all_pairs_redundancy(np.stack([v, -3 * v])), [-1, -1], atol=1e-14)
    # a lone token has redundancy 0, and a zero key has cosine 0 with everything
    np.testing.assert_allclose(O.all_pairs_redundancy(v[None, :]), [0.0])
    z = np.stack([v, np.zeros(d), 2 * v])
    np.testing.assert_allclose(O.all_pairs_redundancy(z), [0.5, 0.0, 0.5], atol=1e-14)


def test_all_pairs_redundancy_brute_force():
    """Pure-Python double loop over the pairs on a small input."""
    rng = np.random.default_rng(13)
    k = rng.standard_normal((11, 5))
    L = k.shape[0]
    want = []
    for t in range(L):
        acc = 0.0
        for j in range(L):
            if j != t:
                dot = sum(float(k[t, e] * k[j, e]) for e in range(5))
                acc += dot / (math.sqrt(sum(float(x * x) for x in k[t])) * math.sqrt(sum(float(x * x) for x in k[j])))
        want.append(acc / (L - 1))
    np.testing.assert_allclose(O.all_pairs_redundancy(k), want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- selection ---------------

def _brute_force_keep(S, k):
    """Independent formulation: t is kept iff fewer than k tokens outrank it."""
    L = len(S)
    s = [(-math.inf if math.isnan(x) else x) for x in S]
    keep = [t for t in range(L)
            if sum(1 for u in range(L) if s[u] > s[t] or (s[u] == s[t] and u < t)) < k]
    return keep


@pytest.mark.parametrize("seed", range(6))
def test_selection_equals_rank_counting(seed):
    rng = np.random.default_rng(seed)
    L = 48
    S = rng.standard_normal(L)
    if seed % 2:
        S = np.round(S * 2) / 2  # many exact ties
    if seed == 5:
        S[[3, 7]] = np.nan
        S[[10, 11]] = np.inf
    for k in (1, 10, 47, 48):
        assert list(O.select_keep(S, k)) == _brute_force_keep(S, k)


def test_selection_tie_keeps_earlier():
    S = np.zeros(8)
    assert list(O.select_keep(S, 5)) == [0, 1, 2, 3, 4]


def test_global_score_dominates_known_keep_set():
    # alpha=1, beta=0, G = 10 * permutation: attn <= 1 cannot reorder, so the kept set is the
    # positions of the k largest G.
    rng = np.random.default_rng(4)
    L, k = 64, 48
    perm = rng.permutation(L)
    G = 10.0 * perm
    attn = rng.dirichlet(np.ones(L))
    R = rng.uniform(-1, 1, L)
    S = O.combine_scores(attn, G, R, 1.0, 0.0, 0, False)
    assert list(O.select_keep(S, k)) == sorted(np.nonzero(perm >= L - k)[0].tolist())


# ---------------------------------------------------------------- whole pass -------------

def _small_llama(**kw):
    from paged_kv_cache_obs_gb300 import synth
    base = dict(num_requests=2, num_layers=2, n_max=8)
    base.update(kw)
    return synth.WORKLOADS["llama3_8b"].scaled(**base)


def _run_pass(wl):
    from paged_kv_cache_obs_gb300 import synth
    inp = synth.make_inputs(wl, "cpu")
    pool = synth.bf16_bits(inp.pool)
    obs_q = synth.bf16_bits(inp.obs_q)
    gs = inp.global_scores.numpy()
    R = inp.num_compress
    tables = inp.block_tables[:R]
    alloc = O.RefcountPool(pool.shape[1])
    for blk, c in enumerate(inp.refcount):
        alloc.refcount[blk] = int(c)
    free = alloc.free_ids()
    dst = tables.copy()
    replaced = []
    for r in range(R):
        row, rep = O.plan_dst_table(tables[r], wl.n_max, dict(enumerate(alloc.refcount)), free)
        dst[r, :wl.n_max - 1] = row
        replaced += rep
    new_pool, new_G, dbg = O.compress_pass(pool, tables, dst, inp.seq_len[:R], inp.qslot, obs_q,
                                           gs, wl.params())
    return inp, pool, obs_q, gs, tables, dst, replaced, new_pool, new_G, dbg


@pytest.mark.parametrize("prefix", [0, 3])
def test_pass_invariants(prefix):
    wl = _small_llama(shared_prefix_blocks=prefix)
    inp, pool, obs_q, gs, tables, dst, replaced, new_pool, new_G, dbg = _run_pass(wl)
    b, L, w = wl.block_size, wl.L, wl.window
    k = (wl.n_max - 1) * b
    for (r, l, h), u in dbg.items():
        src = u["src"]
        assert len(src) == k                                   # exactly k kept
        assert (np.diff(src) > 0).all()                        # original order
        if wl.protect_window:
            assert set(range(L - w, L)) <= set(src.tolist())   # window kept
        assert abs(u["attn"].sum() - 1) < 1e-12
        k_in = O.gather_rows(pool, l, 0, h, tables[r], L, b)
        v_in = O.gather_rows(pool, l, 1, h, tables[r], L, b)
        k_out = O.gather_rows(new_pool, l, 0, h, dst[r], k, b)
        v_out = O.gather_rows(new_pool, l, 1, h, dst[r], k, b)
        assert np.array_equal(k_out, k_in[src]) and np.array_equal(v_out, v_in[src])
        G = gs[r, l, h].astype(np.float64)
        # wiring of the pass: the carried score follows the pinned update rule (hand-worked in
        # test_two_block_hand_example_global_update) on this unit's own kept set and attention
        want_G = O.global_update(G, u["attn"], src, wl.decay, L)
        np.testing.assert_allclose(new_G[r, l, h, :k], want_G[:k].astype(np.float32))
        assert (new_G[r, l, h, k:] == 0).all()
    # shared prefix blocks are byte-identical and replaced by fresh targets
    shared = np.nonzero(inp.refcount > 1)[0]
    assert len(shared) == prefix
    for blk in shared:
        assert np.array_equal(new_pool[:, blk], pool[:, blk])
    assert sorted(set(replaced)) == sorted(shared.tolist())
    assert len(replaced) == prefix * inp.num_compress
    if prefix:
        fresh = dst[:, :prefix]
        assert len(set(fresh.ravel().tolist())) == fresh.size
        assert not set(fresh.ravel().tolist()) & set(np.nonzero(inp.refcount)[0].tolist())


def test_slot_location_hand_example():
    # Paged storage (zh 2.3 "PagedAttention"): logical slot t lives in row t mod b of the block
    # the table names at position t div b.  b = 4, table [7, 3, 9]:
    table = np.array([7, 3, 9])
    assert O.slot_location(table, 0, 4) == (7, 0)
    assert O.slot_location(table, 5, 4) == (3, 1)    # second block, second row
    assert O.slot_location(table, 11, 4) == (9, 3)   # third block, last row


def test_pass_is_per_head_independent():
    # Changing one head's keys changes only that head's selection.
    wl = _small_llama(num_requests=1, num_layers=1, n_max=4)
    from paged_kv_cache_obs_gb300 import synth
    inp = synth.make_inputs(wl, "cpu")
    pool = synth.bf16_bits(inp.pool)
    obs_q = synth.bf16_bits(inp.obs_q)
    gs = inp.global_scores.numpy()
    t = inp.block_tables[:1]
    _, _, d0 = O.compress_pass(pool, t, t, inp.seq_len, inp.qslot, obs_q, gs, wl.params())
    pool2 = pool.copy()
    pool2[0, :, 0, 3] = pool2[0, ::-1, 0, 3]
    _, _, d1 = O.compress_pass(pool2, t, t, inp.seq_len, inp.qslot, obs_q, gs, wl.params())
    for h in range(wl.num_kv_heads):
        same = np.array_equal(d0[(0, 0, h)]["S"], d1[(0, 0, h)]["S"])
        assert same == (h != 3)


# ---------------------------------------------------------------- decode consumer ---------

def test_decode_attention_closed_forms():
    bits = lambda a: O.f64_to_bf16_bits(np.asarray(a, float))
    v = np.array([[1.0, 2.0], [3.0, -4.0]])
    # single key -> its value
    out = O.decode_attention(bits([[1.0, 0.5]]), bits([[2.0, 1.0]]), bits(v[:1]), 0.7)
    np.testing.assert_allclose(out, v[:1], atol=1e-15)
    # logits ln1, ln3 -> weights 1/4, 3/4
    out = O.decode_attention(bits([[1.0, 0.0]]), bits([[0.0, 0.0], [math.log(3), 0.0]]),
                             bits(v), 1.0)
    # ln 3 is rounded to bf16: use the rounded key value in the hand formula
    l3 = O.bf16_bits_to_f64(bits([math.log(3)]))[0]
    w1 = math.exp(l3) / (1 + math.exp(l3))
    np.testing.assert_allclose(out[0], (1 - w1) * v[0] + w1 * v[1], rtol=1e-14)


# ---------------------------------------------------------------- allocator model -------

def test_refcount_pool_model():
    a = O.RefcountPool(6)
    assert a.alloc(2) == [0, 1]
    a.incref([1])
    assert a.alloc(5) is None and a.num_free() == 4
    a.decref([1])
    assert a.refcount[1] == 1
    a.decref([0])
    assert a.alloc(1) == [0]
    table = [1, 0, 2]
    a.incref([1])
    free = a.free_ids()
    dst, rep = O.plan_dst_table(table, 3, dict(enumerate(a.refcount)), free)
    assert dst == [2, 0] and rep == [1]


def test_bf16_round_trip():
    x = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, 65504.0, -1e30])
    bits = O.f64_to_bf16_bits(x)
    back = O.bf16_bits_to_f64(bits)
    assert np.array_equal(O.f64_to_bf16_bits(back), bits)
    assert back[1] == 1.0 and back[2] == -2.5 and back[3] == 3.140625
    # round to nearest even at the halfway point 1 + 2^-8
    assert O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.array([1 + 2 ** -8])))[0] == 1.0


def test_pass_invariants_after_prefill():
    # requests longer than n_max*b (first compression after a long prompt): still exactly k
    # kept per head, the freed slots of the global score zeroed up to the request's length
    from paged_kv_cache_obs_gb300 import synth
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=3, num_layers=1, num_kv_heads=2, num_q_heads=4,
                                            n_max=6, window=8, prefill_max=300)
    inp = synth.make_inputs(wl, "cpu")
    pool = synth.bf16_bits(inp.pool)
    obs_q = synth.bf16_bits(inp.obs_q)
    gs = inp.global_scores.numpy()
    R = inp.num_compress
    t = inp.block_tables[:R]
    new_pool, new_G, dbg = O.compress_pass(pool, t, t, inp.seq_len[:R], inp.qslot, obs_q, gs, wl.params())
    b = wl.block_size
    k = (wl.n_max - 1) * b
    assert (inp.seq_len[:R] > k).all() and (inp.seq_len[:R] <= 300).all()
    for (r, l, h), u in dbg.items():
        L = int(inp.seq_len[r])
        assert len(u["attn"]) == L and len(u["src"]) == k
        assert set(range(L - wl.window, L)) <= set(u["src"].tolist())
        assert (new_G[r, l, h, k:L] == 0).all()
        assert np.array_equal(new_G[r, l, h, L:], gs[r, l, h, L:])   # beyond L untouched
        k_in = O.gather_rows(pool, l, 0, h, t[r], L, b)
        k_out = O.gather_rows(new_pool, l, 0, h, t[r], k, b)
        assert np.array_equal(k_out, k_in[u["src"]])


def test_per_request_budgets_keep_their_own_k():
    # request r keeps (N_max_r - 1) * b tokens per head (per-request budgets)
    from paged_kv_cache_obs_gb300 import synth
    wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=4, num_layers=1, num_kv_heads=2, num_q_heads=4,
                                              n_max=10, window=8, budget_min=2)
    inp = synth.make_inputs(wl, "cpu")
    R = inp.num_compress
    t = inp.block_tables[:R]
    _, new_G, dbg = O.compress_pass(synth.bf16_bits(inp.pool), t, t, inp.seq_len[:R], inp.qslot,
                                    synth.bf16_bits(inp.obs_q), inp.global_scores.numpy(), wl.params(),
                                    n_max_per_req=inp.n_max_req)
    b = wl.block_size
    for (r, l, h), u in dbg.items():
        k_r = (int(inp.n_max_req[r]) - 1) * b
        assert int(inp.seq_len[r]) == int(inp.n_max_req[r]) * b
        assert len(u["src"]) == k_r
        assert (new_G[r, l, h, k_r:int(inp.seq_len[r])] == 0).all()
