"""GPU parity of the compression pass (C-ABI zp_compress) against the CPU oracle.

Small cases compare every unit and every byte of the pool; the full-size workloads run in
the launch configuration the benchmark times and compare sampled units with the oracle plus
size-independent properties of all units.
"""
import numpy as np
import pytest
import torch

from oracle import parity
from oracle import zipage_oracle as O
from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zp():
    from paged_kv_cache_obs_gb300 import build
    import os
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import runner, zipage
    return zipage, runner


def _run(zp, wl, device_gen=False, seed=None, mutate=None):
    zipage, runner = zp
    inp = synth.make_inputs(wl, "cuda" if device_gen else "cpu", seed=seed)
    if mutate:
        mutate(inp)
    pool_in = synth.bf16_bits(inp.pool)
    obs_q = synth.bf16_bits(inp.obs_q)
    gs_in = inp.global_scores.cpu().numpy()
    batch = runner.CompressionBatch(inp, "cuda")
    batch.enable_debug()
    batch.launch()
    err = batch.error()
    torch.cuda.synchronize()
    return inp, batch, pool_in, obs_q, gs_in, err


def _check_all(zp, wl, **kw):
    inp, batch, pool_in, obs_q, gs_in, err = _run(zp, wl, **kw)
    assert err == 0
    R = inp.num_compress
    units = [(r, l, h) for r in range(R) for l in range(wl.num_layers) for h in range(wl.num_kv_heads)]
    dbg = {k: v.cpu().numpy() for k, v in batch.debug.items()}
    ndiff = parity.check_units(units, pool_in, obs_q, gs_in, batch.tables, batch.dst_tables,
                               inp.seq_len[:R], inp.qslot, wl.params(), dbg,
                               batch.gs.cpu().numpy(), synth.bf16_bits(batch.pool), full_pool=True,
                               n_max_per_req=inp.n_max_req)
    batch.close()
    return ndiff


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "qwen2_small": synth.WORKLOADS["qwen2_7b"].scaled(num_requests=2, num_layers=2),
    "llama3_small": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2),
    "prefix_small": synth.WORKLOADS["shared_prefix"].scaled(num_requests=3, num_layers=2),
    # L = 1152: five CTAs, the last one holds a ragged 128 keys
    "ragged_cluster": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2, n_max=72),
    # L = 144: one CTA whose second key half holds 16 keys
    "ragged_cta": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, n_max=9, window=8),
    # d = 64 with b = 32 and L = 320: two CTAs, 64 keys in the second
    "d64_b32": synth.WORKLOADS["tiny"].scaled(num_requests=2, num_layers=2, num_q_heads=8,
                                              num_kv_heads=2, block_size=32, n_max=10, window=4,
                                              global_init="uniform"),
    "no_protect_noncausal": synth.WORKLOADS["llama3_8b"].scaled(num_requests=1, num_layers=2, n_max=16,
                                                                protect_window=0, causal=0),
    "one_window_row": synth.WORKLOADS["qwen2_7b"].scaled(num_requests=1, num_layers=1, n_max=8, window=1),
    # first compression after a prefill: L in (k, 1100], k = 496, so E spans 1..604 (both
    # selection paths), partial last blocks, and CTAs past a short request's end
    "prefill_small": synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=2, n_max=32, prefill_max=1100),
    "prefill_d64_b32": synth.WORKLOADS["tiny"].scaled(num_requests=3, num_layers=2, num_q_heads=8, num_kv_heads=2,
                                                      block_size=32, n_max=10, window=4, prefill_max=700,
                                                      global_init="uniform"),
    "prefill_one_cta": synth.WORKLOADS["prefill"].scaled(num_requests=3, num_layers=1, n_max=9, window=8,
                                                         prefill_max=250),
    # per-request budgets N_max_r in 3..40, each request at its own trigger (N_max_r full blocks):
    # clusters of 1..3 active CTAs under a launch of 3
    "budgets_small": synth.WORKLOADS["llama3_8b"].scaled(num_requests=5, num_layers=2, n_max=40, window=16,
                                                         budget_min=3),
    # beyond one portable cluster: 16-CTA clusters (one CTA per SM).  A decode trigger at
    # L = 3200 (13 CTAs, E = 16), and long prefills (L = 1171 .. 3824 in a launch of 16 CTAs,
    # E up to 2816)
    "long_trigger": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, num_kv_heads=2,
                                                        num_q_heads=8, n_max=200),
    "long_prefill": synth.WORKLOADS["prefill"].scaled(num_requests=6, num_layers=1, num_kv_heads=2,
                                                      num_q_heads=8, n_max=64, prefill_max=4000),
    # beyond one cluster: the multi-pass form (launch length above 4096).  Long prefills up to
    # 9000 tokens (E up to about 8000), and a decode trigger at L = 4800 (N_max = 300, E = 16)
    "multipass_prefill": synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=1, num_kv_heads=2,
                                                           num_q_heads=8, n_max=64, prefill_max=9000),
    "multipass_trigger": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, num_kv_heads=2,
                                                             num_q_heads=8, n_max=300),
    # the multi-pass form with d = 64 and b = 32 (one 64-column half, two 8-row groups per
    # block), and with the Qwen2 grouping G_q = 7 (w = 16: 112 window rows, 16 padding rows of
    # the MMA) at a decode trigger of L = 5120
    "multipass_d64_b32": synth.WORKLOADS["tiny"].scaled(num_requests=3, num_layers=1, num_q_heads=8, num_kv_heads=2,
                                                        block_size=32, n_max=20, window=4, prefill_max=6000,
                                                        global_init="uniform"),
    "multipass_gq7": synth.WORKLOADS["qwen2_7b"].scaled(num_requests=1, num_layers=1, num_q_heads=14,
                                                        num_kv_heads=2, n_max=160),
    # the multi-pass compaction computes its row offsets 256 slots at a time: k = 4096 kept
    # slots end exactly on such a group (L = 4112, E = 16)
    "multipass_k_on_group": synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, num_kv_heads=2,
                                                                num_q_heads=8, n_max=257),
    # the multi-pass form with per-request budgets (N_max_r in 200..300, so L_r = 3200..4800
    # on both sides of one cluster's 4096 keys) and with shared prefix blocks that the plan
    # replaces by target blocks
    "multipass_budgets": synth.WORKLOADS["llama3_8b"].scaled(num_requests=4, num_layers=1, num_kv_heads=2,
                                                             num_q_heads=8, n_max=300, budget_min=200),
    "multipass_prefix": synth.WORKLOADS["shared_prefix"].scaled(num_requests=3, num_layers=1, num_kv_heads=2,
                                                                num_q_heads=8, n_max=300),
    # shared prefix blocks with lengths that differ (the grouped launches of the fused pass), and
    # with 16-CTA clusters
    "prefill_prefix": synth.WORKLOADS["shared_prefix"].scaled(num_requests=4, num_layers=1, num_kv_heads=2,
                                                              num_q_heads=8, n_max=32, prefill_max=1500),
    "long_prefix": synth.WORKLOADS["shared_prefix"].scaled(num_requests=2, num_layers=1, num_kv_heads=2,
                                                           num_q_heads=8, n_max=200),
    # per-request budgets from 20 to 200 blocks: length groups of 2 to 13 CTAs in one call, so
    # both cluster widths (up to 8, and 16) run side by side
    "long_budgets": synth.WORKLOADS["llama3_8b"].scaled(num_requests=6, num_layers=1, num_kv_heads=2,
                                                        num_q_heads=8, n_max=200, budget_min=20),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_compress_matches_oracle_every_unit(zp, name):
    ndiff = _check_all(zp, SMALL[name])
    assert ndiff <= 2


@pytest.mark.parametrize("path", ["trigger", "many_evictions", "multipass"])
def test_exact_ties_keep_the_earlier_tokens(zp, path):
    # all keys of a head identical, no global score, alpha = beta = 0, non-causal: every
    # unprotected token has the same score, so the earliest k tokens are kept.  The paths:
    # E = b at the decode trigger; E up to 632 after a prefill (ranks across the cluster);
    # a launch length past 4096 (radix select, which must resolve the ties by position).
    kw = dict(num_requests=1, num_layers=1, n_max=24, alpha=0.0, beta=0.0, causal=0, protect_window=0)
    if path == "trigger":
        wl = synth.WORKLOADS["llama3_8b"].scaled(**kw)
    else:
        wl = synth.WORKLOADS["prefill"].scaled(num_kv_heads=2, num_q_heads=8,
                                               prefill_max=1000 if path == "many_evictions" else 5000, **kw)

    def mutate(inp):
        inp.pool[:, :, 0] = inp.pool[:, :1, 0, :, :1]

    inp, batch, pool_in, obs_q, gs_in, err = _run(zp, wl, mutate=mutate)
    assert err == 0
    k = (wl.n_max - 1) * wl.block_size
    keep = batch.debug["keep"].cpu().numpy()[0, 0]
    for h in range(wl.num_kv_heads):
        assert np.array_equal(np.nonzero(keep[h])[0], np.arange(k))
    batch.close()


def test_lowest_scores_fill_whole_ctas(zp):
    # first compressions after a prefill (E up to 972) whose 256 lowest scores are the keys of
    # one CTA (CTA 0 for even heads, CTA 1 for odd ones): every kept key then ranks above the
    # whole sorted list of that CTA, and its rank must count all 256 of them
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=6, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                           n_max=9, window=8, prefill_max=1100)

    def mutate(inp):
        assert sum(int(x) >= 128 + 512 for x in inp.seq_len) >= 2  # both CTAs full, E >= 256
        for h in range(wl.num_kv_heads):
            lo = 256 * (h % 2)
            inp.global_scores[:, :, h, lo:lo + 256] = -10.0

    ndiff = _check_all(zp, wl, mutate=mutate)
    assert ndiff == 0


def test_eviction_counts_at_the_path_boundaries(zp):
    # one launch whose requests evict exactly E = 1, 31, 32 (the last few-eviction case), 33
    # (the first many-eviction case), 256 and 257 tokens per head: each request's length is
    # cut to k + E inside the blocks it already holds
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=6, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                           n_max=9, window=8, prefill_max=1100)
    k = (wl.n_max - 1) * wl.block_size

    def mutate(inp):
        order = np.argsort(inp.seq_len[:6], kind="stable")
        for r, e in zip(order, [1, 31, 32, 33, 256, 257]):
            assert int(inp.seq_len[r]) >= k + e
            inp.seq_len[r] = k + e

    assert _check_all(zp, wl, mutate=mutate) == 0


def test_maximum_length_multipass(zp):
    # the longest sequences the library takes (L = 16384, the multi-pass form): a decode trigger
    # (E = 16) and, through a per-request budget of 64 blocks, a prefill-sized eviction
    # (E = 16384 - 1008 = 15376) in the same launch
    wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                             n_max=1024)

    def mutate(inp):
        assert (inp.seq_len[:2] == 16384).all()
        inp.n_max_req = np.array([1024, 64], dtype=np.int32)

    assert _check_all(zp, wl, mutate=mutate) <= 2


def test_bad_block_id_skips_the_request_and_reports(zp):
    wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2, n_max=16)
    zipage, runner = zp
    inp = synth.make_inputs(wl, "cpu")
    pool_in = synth.bf16_bits(inp.pool)
    batch = runner.CompressionBatch(inp, "cuda")
    bad = batch.d_tables.clone()
    bad[1, 3] = inp.pool.shape[1] + 5  # request 1 points outside the pool
    batch.d_tables = bad
    batch.launch()
    assert batch.error() == zipage.ZP_ERR_BAD_TABLE
    out = synth.bf16_bits(batch.pool)
    # request 1's blocks are untouched; request 0 was compressed
    for blk in inp.block_tables[1, :wl.n_max]:
        assert np.array_equal(out[:, blk], pool_in[:, blk])
    assert not np.array_equal(out[:, inp.block_tables[0, :wl.n_max - 1]],
                              pool_in[:, inp.block_tables[0, :wl.n_max - 1]])
    batch.close()


def test_unsupported_and_empty_calls(zp):
    zipage, runner = zp
    wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=1, num_layers=1, n_max=8)
    inp = synth.make_inputs(wl, "cpu")
    batch = runner.CompressionBatch(inp, "cuda")
    with pytest.raises(zipage.ZipageError) as e:   # n_max = 160 is wider than the 8-entry tables
        zipage.zp_compress(batch.pool, batch.d_tables, batch.d_seq, batch.d_qslot, batch.d_dst,
                           batch.obs_q, batch.gs, dict(batch.params, n_max=160), batch.workspace)
    assert e.value.status in (zipage.ZP_ERR_UNSUPPORTED, zipage.ZP_ERR_INVALID_ARG)
    with pytest.raises(zipage.ZipageError) as e:   # w*G_q = 33*4 > 128 window rows
        zipage.zp_compress(batch.pool, batch.d_tables, batch.d_seq, batch.d_qslot, batch.d_dst,
                           batch.obs_q, batch.gs, dict(batch.params, window=33), batch.workspace)
    assert e.value.status == zipage.ZP_ERR_UNSUPPORTED
    before = synth.bf16_bits(batch.pool)
    zipage.zp_compress(batch.pool, batch.d_tables[:0], batch.d_seq[:0], batch.d_qslot[:0],
                       batch.d_dst[:0], batch.obs_q, batch.gs, batch.params, batch.workspace)
    torch.cuda.synchronize()
    assert np.array_equal(before, synth.bf16_bits(batch.pool))
    batch.close()


@pytest.mark.parametrize("path", ["one_size", "grouped"])
@pytest.mark.parametrize("bad_len", ["no_eviction", "too_long"])
def test_wrong_seq_len_is_reported(zp, bad_len, path):
    # "grouped": the launch length (600) is above n_max*b, so the requests are grouped by
    # length and a request whose length is invalid must still reach a kernel that reports it
    zipage, runner = zp
    if path == "one_size":
        wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=1, n_max=8)
    else:
        wl = synth.WORKLOADS["prefill"].scaled(num_requests=3, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                               n_max=8, prefill_max=600)
    inp = synth.make_inputs(wl, "cpu")
    pool_in = synth.bf16_bits(inp.pool)
    batch = runner.CompressionBatch(inp, "cuda")
    La = batch.max_seq_len or wl.L
    # a request must hold more than k = (n_max-1)*b tokens and at most the launch length
    batch.d_seq[0] = (wl.n_max - 1) * wl.block_size if bad_len == "no_eviction" else La + 1
    batch.launch()
    assert batch.error() == zipage.ZP_ERR_BAD_TABLE
    out = synth.bf16_bits(batch.pool)
    for blk in inp.block_tables[0, :wl.n_max]:
        assert np.array_equal(out[:, blk], pool_in[:, blk])
    batch.close()


# ------------------------------------------------------------------ full-size workloads -----

FULL = ["qwen2_7b", "llama3_8b", "shared_prefix", "prefill", "prefill_long"]


def _compaction_property_all_units(batch, pristine, keep):
    """Every unit: compacted row j equals input row src_j (bit-exact), k kept per head,
    protected window kept; blocks outside the destination tables are unchanged."""
    wl = batch.wl
    b, k, w = wl.block_size, (wl.n_max - 1) * wl.block_size, wl.window
    nl, Hkv = wl.num_layers, wl.num_kv_heads
    counts = keep.sum(-1)
    assert bool((counts == k).all())
    dev = batch.pool.device
    li = torch.arange(nl, device=dev)[:, None, None]
    hi = torch.arange(Hkv, device=dev)[None, :, None]
    for r in range(batch.inp.num_compress):
        L = int(batch.seq_len[r])
        if wl.protect_window:
            assert bool((keep[r, ..., L - w:L] == 1).all())
        assert bool((keep[r, ..., L:] == 0).all())
        pos = torch.arange(L, device=dev)
        src = pos.expand(nl, Hkv, L)[keep[r, ..., :L].bool()].view(nl, Hkv, k)
        tab = torch.from_numpy(batch.tables[r]).to(dev).long()
        dtab = torch.from_numpy(batch.dst_tables[r]).to(dev).long()
        j = torch.arange(k, device=dev)
        for kv in (0, 1):
            old = pristine[li, tab[src // b], kv, hi, src % b]
            new = batch.pool[li, dtab[j // b][None, None, :], kv, hi, (j % b)[None, None, :]]
            assert torch.equal(old.view(torch.int16), new.view(torch.int16)), f"request {r} kv {kv}"
    written = set(batch.dst_tables[:, :wl.n_max - 1].ravel().tolist())
    written.discard(-1)
    others = torch.tensor(sorted(set(range(batch.pool.shape[1])) - written), device=dev)
    assert torch.equal(pristine[:, others].view(torch.int16), batch.pool[:, others].view(torch.int16))


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_units_and_properties(zp, name):
    zipage, runner = zp
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda")
    pristine = inp.pool.clone()
    gs_in = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    batch.enable_debug()
    batch.launch()
    assert batch.error() == 0
    keep = batch.debug["keep"]
    _compaction_property_all_units(batch, pristine, keep)
    check_sampled_units(batch, inp, pristine, gs_in, seed=7)
    # shared prefix blocks are byte-identical
    shared = np.nonzero(inp.refcount > 1)[0]
    if len(shared):
        sb = torch.tensor(shared, device="cuda")
        assert torch.equal(pristine[:, sb].view(torch.int16), batch.pool[:, sb].view(torch.int16))
    batch.close()


def check_sampled_units(batch, inp, pristine, gs_in, seed, n=6):
    """n seeded random units plus the first and the last unit of a full-size launch, checked
    against the oracle on the sampled requests' blocks (debug outputs, global scores and the
    compacted rows)."""
    wl = inp.wl
    rng = np.random.default_rng(seed)
    R = inp.num_compress
    units = [(int(rng.integers(R)), int(rng.integers(wl.num_layers)), int(rng.integers(wl.num_kv_heads)))
             for _ in range(n)] + [(0, 0, 0), (R - 1, wl.num_layers - 1, wl.num_kv_heads - 1)]
    units = sorted(set(units))
    reqs = sorted({u[0] for u in units})
    # oracle inputs restricted to the sampled requests (their blocks only)
    sub_tables = batch.tables[reqs]
    sub_dst = batch.dst_tables[reqs]
    blocks = sorted((set(sub_tables.ravel().tolist()) | set(sub_dst.ravel().tolist())) - {-1})
    remap = {blk: i for i, blk in enumerate(blocks)}
    remap[-1] = -1
    rt = np.vectorize(remap.get)(sub_tables).astype(np.int32)
    rd = np.vectorize(remap.get)(sub_dst).astype(np.int32)
    bidx = torch.tensor(blocks, device="cuda")
    pool_in = synth.bf16_bits(pristine[:, bidx])
    pool_out = synth.bf16_bits(batch.pool[:, bidx])
    qs = torch.tensor(inp.qslot[reqs], device="cuda").long()
    obs_q = synth.bf16_bits(batch.obs_q[qs])
    gsi = gs_in[qs].cpu().numpy()
    gso = batch.gs[qs].cpu().numpy()
    dbg = {k: v[torch.tensor(reqs, device="cuda")].cpu().numpy() for k, v in batch.debug.items()}
    ridx = {r: i for i, r in enumerate(reqs)}
    sub_units = [(ridx[r], l, h) for (r, l, h) in units]
    p = wl.params()
    ndiff = parity.check_units(sub_units, pool_in, obs_q, gsi, rt, rd, inp.seq_len[reqs],
                               np.arange(len(reqs), dtype=np.int32), p, dbg, gso, pool_out)
    assert ndiff <= 2


@pytest.mark.parametrize("name", ["llama3_8b", "prefill"])
def test_timed_launch_without_debug_outputs_is_bit_identical(zp, name):
    """The benchmark times zp_compress without the per-token debug outputs, a launch in which
    the kernel skips those stores.  From the same pristine state, that launch must leave every
    pool byte and every global score bit-identical to a launch with the outputs on, which is
    itself checked against the oracle here (sampled units and all-unit properties)."""
    zipage, runner = zp
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, "cuda")
    pristine = inp.pool.clone()
    gs_in = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    batch.enable_debug()
    batch.launch()
    assert batch.error() == 0
    _compaction_property_all_units(batch, pristine, batch.debug["keep"])
    check_sampled_units(batch, inp, pristine, gs_in, seed=11, n=3)
    pool_dbg, gs_dbg = batch.pool.clone(), batch.gs.clone()
    batch.pool.copy_(pristine)
    batch.gs.copy_(gs_in)
    batch.debug = None
    stream = torch.cuda.Stream()          # as the benchmark launches it
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        batch.launch(stream=stream)
    assert batch.error(stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(batch.pool.view(torch.int16), pool_dbg.view(torch.int16))
    assert torch.equal(batch.gs.view(torch.int32), gs_dbg.view(torch.int32))
    batch.close()


@pytest.mark.parametrize("grouped", [False, True])
def test_layer_by_layer_equals_one_call(zp, grouped):
    """Compressing the layers one call at a time, in any order, gives the same bytes as one
    call over every layer (units are independent; the one-call pass is checked against the
    oracle by the tests above).  "grouped": requests of different lengths after a prefill, so
    every call groups them by cluster size again."""
    zipage, runner = zp
    if grouped:
        wl = synth.WORKLOADS["prefill"].scaled(num_requests=5, num_layers=4, num_kv_heads=2, num_q_heads=8,
                                               n_max=16, prefill_max=1500)
    else:
        wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=4)
    inp = synth.make_inputs(wl, "cpu", seed=77)
    whole = runner.CompressionBatch(inp, "cuda")
    whole.launch()
    assert whole.error() == 0
    parts = runner.CompressionBatch(inp, "cuda")
    for layer in (2, 0, 3, 1):
        parts.launch(layers=(layer, 1))
        assert parts.error() == 0
    torch.cuda.synchronize()
    assert torch.equal(parts.pool.view(torch.int16), whole.pool.view(torch.int16))
    assert torch.equal(parts.gs, whole.gs)
    with pytest.raises(zipage.ZipageError):
        parts.launch(layers=(3, 2))  # past the last layer
    whole.close()
    parts.close()


def _random_config(seed):
    """A seeded random small configuration inside the library's limits: d in {64, 128},
    b in {16, 32}, G_q in {1, 2, 4, 7, 8}, w with w*G_q <= 128 and w <= k, budgets, prefill
    lengths (one or several CTAs, or the multi-pass form), shared leading blocks, masks and
    weights."""
    rng = np.random.default_rng(seed)
    d = int(rng.choice([64, 128]))
    b = int(rng.choice([16, 32]))
    gq = int(rng.choice([1, 2, 4, 7, 8]))
    hkv = int(rng.choice([1, 2]))
    n_max = int(rng.integers(3, 41))
    k = (n_max - 1) * b
    w = int(rng.integers(1, min(128 // gq, k) + 1))
    kind = rng.choice(["trigger", "prefill", "budgets", "prefix"])
    kw = dict(num_requests=int(rng.integers(1, 4)), num_layers=int(rng.integers(1, 3)), num_q_heads=gq * hkv,
              num_kv_heads=hkv, head_dim=d, block_size=b, n_max=n_max, window=w,
              key_recipe=str(rng.choice(["normal", "clustered", "rope"])), global_init="uniform",
              alpha=float(rng.uniform(0, 1)), beta=float(rng.uniform(0, 1)), decay=float(rng.uniform(0.5, 1)),
              protect_window=int(rng.integers(0, 2)), causal=int(rng.integers(0, 2)))
    if kind == "prefill":
        kw["prefill_max"] = int(rng.choice([k + 2 * b, 2 * n_max * b, 4500, 6000]))
    elif kind == "budgets" and n_max > 3:
        kw["budget_min"] = 3
    elif kind == "prefix" and n_max > 4:
        kw["shared_prefix_blocks"] = int(rng.integers(1, n_max - 2))
    return synth.WORKLOADS["tiny"].scaled(**kw)


@pytest.mark.parametrize("seed", range(48))
def test_random_configurations_match_oracle(zp, seed):
    wl = _random_config(1000 + seed)
    assert _check_all(zp, wl) <= 2, wl


BAD_KINDS = ["src_past_pool", "src_negative", "dst_past_pool", "qslot_past_slots", "qslot_negative"]


@pytest.mark.parametrize("path", ["fused", "grouped", "multipass"])
@pytest.mark.parametrize("kind", BAD_KINDS)
def test_bad_metadata_skips_only_that_request(zp, kind, path):
    # request 1 carries one bad entry: the call reports ZP_ERR_BAD_TABLE, request 1's blocks and
    # global scores stay as they were, and request 0 is compressed exactly as the oracle says
    zipage, runner = zp
    if path == "fused":
        wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2, num_kv_heads=2, num_q_heads=8,
                                                 n_max=16)
    elif path == "grouped":  # k = 240, lengths up to 1000: clusters of 1 to 4 CTAs
        wl = synth.WORKLOADS["prefill"].scaled(num_requests=2, num_layers=2, num_kv_heads=2, num_q_heads=8,
                                               n_max=16, prefill_max=1000)
    else:
        wl = synth.WORKLOADS["prefill"].scaled(num_requests=2, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                               n_max=64, prefill_max=5000)
    inp = synth.make_inputs(wl, "cpu")
    pool_in = synth.bf16_bits(inp.pool)
    gs_in = inp.global_scores.numpy().copy()
    batch = runner.CompressionBatch(inp, "cuda")
    batch.enable_debug()
    NB = inp.pool.shape[1]
    if kind.startswith("src"):
        t = batch.d_tables.clone()
        t[1, 2] = NB + 5 if kind == "src_past_pool" else -3
        batch.d_tables = t
    elif kind == "dst_past_pool":
        t = batch.d_dst.clone()
        t[1, 1] = NB + 7
        batch.d_dst = t
    else:
        q = batch.d_qslot.clone()
        q[1] = inp.obs_q.shape[0] + 2 if kind == "qslot_past_slots" else -1
        batch.d_qslot = q
    batch.launch()
    assert batch.error() == zipage.ZP_ERR_BAD_TABLE
    torch.cuda.synchronize()
    out = synth.bf16_bits(batch.pool)
    L1 = int(inp.seq_len[1])
    blocks1 = set(inp.block_tables[1, :(L1 + wl.block_size - 1) // wl.block_size].tolist())
    blocks1 |= set(batch.dst_tables[1, :wl.n_max - 1].tolist())
    for blk in blocks1:
        assert np.array_equal(out[:, blk], pool_in[:, blk]), blk
    assert np.array_equal(batch.gs.cpu().numpy()[1], gs_in[1])
    # request 0 against the oracle, unit by unit
    dbg = {k: v.cpu().numpy() for k, v in batch.debug.items()}
    units = [(0, l, h) for l in range(wl.num_layers) for h in range(wl.num_kv_heads)]
    ndiff = parity.check_units(units, pool_in, synth.bf16_bits(inp.obs_q), gs_in, batch.tables, batch.dst_tables,
                               inp.seq_len[:2], inp.qslot, wl.params(), dbg, batch.gs.cpu().numpy(), out)
    assert ndiff <= 2
    batch.close()


@pytest.mark.parametrize("R,n_max,prefill_max", [(37, 16, 2048), (600, 8, 600)])
def test_length_groups_partition_the_requests(zp, R, n_max, prefill_max):
    # After a call whose requests need different cluster sizes, the workspace holds the
    # grouping it ran: group c (c CTAs of 256 keys) starts at int 48 + 2c of the header with
    # (first position, count), and the order follows the 512-byte header.  Every request is in
    # exactly one group, the group of ceil(L/256) CTAs, in request order.  600 requests give
    # the grouping kernel's threads several requests each.
    zipage, runner = zp
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=R, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                           n_max=n_max, prefill_max=prefill_max)
    inp = synth.make_inputs(wl, "cpu")
    batch = runner.CompressionBatch(inp, "cuda")
    k = (n_max - 1) * wl.block_size
    c_lo, c_hi = (k + 1 + 255) // 256, (prefill_max + 255) // 256
    assert zipage.zp_compress_kernel_launches(batch.params, batch.max_seq_len) == 1 + (c_hi - c_lo + 1)
    batch.launch()
    assert batch.error() == 0
    torch.cuda.synchronize()
    assert inp.num_compress == R
    ws = batch.workspace.view(torch.int32).cpu().numpy()
    order = ws[128:128 + R]
    seen = []
    for c in range(c_lo, c_hi + 1):
        start, count = int(ws[48 + 2 * c]), int(ws[48 + 2 * c + 1])
        members = order[start:start + count].tolist()
        assert members == sorted(members)
        for r in members:
            assert (int(inp.seq_len[r]) + 255) // 256 == c
        seen += members
    assert sorted(seen) == list(range(R))
    batch.close()
