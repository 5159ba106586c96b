"""GPU parity of paged decode attention (zp_paged_decode_attn) and of the mixed serving step:
compression on a side stream while decode runs on the main stream."""
import numpy as np
import pytest
import torch

from oracle import parity
from oracle import zipage_oracle as O
from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu

# bf16 output: rounding is at most 2^-9 relative; fp32 accumulation adds far less
DEC_RTOL, DEC_ATOL = 4e-3, 1e-4


@pytest.fixture(scope="module")
def zp():
    import os
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import runner, zipage
    return zipage, runner


def _decode_case(zipage, Hq, Hkv, d, b, seq_lens, layers=2, seed=0, layer=1):
    g = torch.Generator().manual_seed(seed)
    B = len(seq_lens)
    max_blocks = max((s + b - 1) // b for s in seq_lens) + 1
    NB = B * max_blocks + 7
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g).to(torch.bfloat16)
    perm = torch.randperm(NB, generator=g).numpy().astype(np.int32)
    tables = perm[:B * max_blocks].reshape(B, max_blocks).copy()
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16)
    p = dict(num_layers=layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=max_blocks,
             window=1, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    dp, dq = pool.cuda(), q.cuda()
    dt = torch.from_numpy(tables).cuda()
    ds = torch.tensor(seq_lens, dtype=torch.int32).cuda()
    out = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, B, max_blocks))
    zipage.zp_paged_decode_attn(dp, layer, dq, dt, ds, out, p, ws)
    assert zipage.zp_read_error(ws) == 0
    got = O.bf16_bits_to_f64(synth.bf16_bits(out))
    pb, qb = synth.bf16_bits(pool), synth.bf16_bits(q)
    G = Hq // Hkv
    for r, s in enumerate(seq_lens):
        for h in range(Hkv):
            k = O.gather_rows(pb, layer, 0, h, tables[r], s, b)
            v = O.gather_rows(pb, layer, 1, h, tables[r], s, b)
            want = O.decode_attention(qb[r, h * G:(h + 1) * G], k, v, p["scale"])
            err = np.abs(got[r, h * G:(h + 1) * G] - want)
            assert (err <= DEC_RTOL * np.abs(want) + DEC_ATOL).all(), (r, h, float(err.max()))


@pytest.mark.parametrize("Hq,Hkv,d,b", [(32, 8, 128, 16), (28, 4, 128, 32), (8, 8, 64, 16), (16, 2, 64, 32),
                                        (8, 4, 128, 16)])
def test_decode_matches_oracle(zp, Hq, Hkv, d, b):
    zipage, _ = zp
    _decode_case(zipage, Hq, Hkv, d, b, [1, b - 1, b, b + 1, 255, 256, 257, 700])


@pytest.mark.parametrize("seed", range(16))
def test_decode_random_configurations(zp, seed):
    # seeded shapes and lengths: G_q in {1, 2, 4, 7, 8}, d in {64, 128}, b in {16, 32}, batches
    # of 1..9 requests with lengths from 1 token to several splits (split = 32 blocks)
    zipage, _ = zp
    rng = np.random.default_rng(2000 + seed)
    g = int(rng.choice([1, 2, 4, 7, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    d, b = int(rng.choice([64, 128])), int(rng.choice([16, 32]))
    lens = [int(x) for x in rng.integers(1, int(rng.choice([64, 600, 3000])) + 1, size=int(rng.integers(1, 10)))]
    _decode_case(zipage, g * hkv, hkv, d, b, lens, layers=int(rng.integers(1, 3)), seed=seed, layer=0)


def test_decode_long_sequences_many_splits(zp):
    zipage, _ = zp
    _decode_case(zipage, 32, 8, 128, 16, [2048, 2047, 1500, 33], seed=3)


def test_decode_bad_block_id_reports(zp):
    zipage, _ = zp
    p = dict(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16, n_max=4, window=1,
             alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    pool = torch.zeros((1, 8, 2, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    tables = torch.tensor([[0, 1, 99, 2]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([50], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, 1, 4))
    zipage.zp_paged_decode_attn(pool, 0, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == zipage.ZP_ERR_BAD_TABLE


@pytest.mark.parametrize("bad_seq", [0, -4, 4 * 16 + 1])
def test_decode_bad_seq_len_reports_and_keeps_the_others(zp, bad_seq):
    # request 1's length is outside 1 .. max_blocks*b: the call reports it and leaves its output
    # untouched; requests 0 and 2 are decoded as the oracle says
    zipage, _ = zp
    g = torch.Generator().manual_seed(5)
    p = dict(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16, n_max=4, window=1,
             alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    pool = torch.randn((1, 12, 2, 2, 16, 64), generator=g).to(torch.bfloat16)
    tables = torch.tensor([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]], dtype=torch.int32)
    seq = torch.tensor([37, bad_seq, 64], dtype=torch.int32)
    q = torch.randn((3, 4, 64), generator=g).to(torch.bfloat16)
    out = torch.full((3, 4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, 3, 4))
    zipage.zp_paged_decode_attn(pool.cuda(), 0, q.cuda(), tables.cuda(), seq.cuda(), out, p, ws)
    assert zipage.zp_read_error(ws) == zipage.ZP_ERR_BAD_TABLE
    got = out.float().cpu()
    assert bool((got[1] == 7.0).all())
    pb, qb = synth.bf16_bits(pool), synth.bf16_bits(q)
    for r in (0, 2):
        for h in range(2):
            k = O.gather_rows(pb, 0, 0, h, tables[r].numpy(), int(seq[r]), 16)
            v = O.gather_rows(pb, 0, 1, h, tables[r].numpy(), int(seq[r]), 16)
            want = O.decode_attention(qb[r, 2 * h:2 * h + 2], k, v, p["scale"])
            err = np.abs(got[r, 2 * h:2 * h + 2].numpy() - want)
            assert (err <= DEC_RTOL * np.abs(want) + DEC_ATOL).all(), (r, h)


def test_mixed_step_side_stream(zp):
    """Compression of the slot holders on a side stream, decode of the others on the main
    stream, then the event-deferred release of the last blocks."""
    zipage, runner = zp
    wl = synth.WORKLOADS["mixed"].scaled(num_requests=4, num_layers=3, num_decode=12)
    inp = synth.make_inputs(wl, "cpu")
    pool_in = synth.bf16_bits(inp.pool)
    obs_q = synth.bf16_bits(inp.obs_q)
    gs_in = inp.global_scores.numpy()
    R = inp.num_compress
    batch = runner.CompressionBatch(inp, "cuda")
    batch.enable_debug()
    p = wl.params()
    dec_tables = torch.from_numpy(np.ascontiguousarray(inp.block_tables[R:])).cuda()
    dec_seq = torch.from_numpy(np.ascontiguousarray(inp.seq_len[R:])).cuda()
    nd = wl.num_decode
    dq = inp.decode_q.cuda()
    outs = torch.zeros((wl.num_layers, nd, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = [zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, nd, wl.n_max)) for _ in range(wl.num_layers)]
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    free_before = zipage.zp_num_free(batch.alloc)
    with torch.cuda.stream(side):
        batch.launch(stream=side)
        batch.commit(stream=side)       # last blocks released only when the side stream is done
    for l in range(wl.num_layers):
        zipage.zp_paged_decode_attn(batch.pool, l, dq[l], dec_tables, dec_seq, outs[l], p, ws[l], stream=main)
    assert zipage.zp_num_pending(batch.alloc) >= 0
    side.synchronize()
    main.synchronize()
    zipage.zp_alloc_drain(batch.alloc)
    assert zipage.zp_num_pending(batch.alloc) == 0
    assert zipage.zp_num_free(batch.alloc) == free_before + R
    assert batch.error(stream=side) == 0
    for w_ in ws:
        assert zipage.zp_read_error(w_) == 0
    # decode results: the decode requests' blocks are disjoint from the compressing ones
    got = O.bf16_bits_to_f64(synth.bf16_bits(outs))
    qb = synth.bf16_bits(inp.decode_q)
    G = wl.num_q_heads // wl.num_kv_heads
    for l in range(wl.num_layers):
        for i in range(nd):
            r = R + i
            s = int(inp.seq_len[r])
            for h in range(wl.num_kv_heads):
                k = O.gather_rows(pool_in, l, 0, h, inp.block_tables[r], s, wl.block_size)
                v = O.gather_rows(pool_in, l, 1, h, inp.block_tables[r], s, wl.block_size)
                want = O.decode_attention(qb[l, i, h * G:(h + 1) * G], k, v, wl.scale)
                err = np.abs(got[l, i, h * G:(h + 1) * G] - want)
                assert (err <= DEC_RTOL * np.abs(want) + DEC_ATOL).all()
    # compression results, every unit and every pool byte
    units = [(r, l, h) for r in range(R) for l in range(wl.num_layers) for h in range(wl.num_kv_heads)]
    dbg = {k: v.cpu().numpy() for k, v in batch.debug.items()}
    parity.check_units(units, pool_in, obs_q, gs_in, batch.tables, batch.dst_tables, inp.seq_len[:R],
                       inp.qslot, p, dbg, batch.gs.cpu().numpy(), synth.bf16_bits(batch.pool), full_pool=True)
    batch.close()


def test_mixed_step_full_size(zp):
    """The mixed serving step at its stated size, run as the benchmark runs it: the 32 slot
    holders (128 full blocks each) compress on a side stream while decode attention of the 224
    other requests (U{1..128} blocks) runs for all 32 layers on a high-priority stream, with the
    split size each decode call chooses.  The pool holds the blocks in use.  Checked: the
    compaction of every compressed unit (kept count, window, bit-exact rows, untouched blocks),
    sampled compression units against the oracle, and sampled decode outputs against the oracle
    (first and last layer, the shortest and longest requests, seeded random others)."""
    from test_gpu_compress import _compaction_property_all_units, check_sampled_units
    zipage, runner = zp
    wl = synth.WORKLOADS["mixed"]
    inp = synth.make_inputs(wl, "cuda")
    R, nd, nl = inp.num_compress, wl.num_decode, wl.num_layers
    assert (R, nd, nl) == (32, 224, 32)
    pristine = inp.pool.clone()
    gs_in = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    batch.enable_debug()
    p = wl.params()
    dec_tables = torch.from_numpy(np.ascontiguousarray(inp.block_tables[R:])).cuda()
    dec_seq = torch.from_numpy(np.ascontiguousarray(inp.seq_len[R:])).cuda()
    outs = torch.zeros((nl, nd, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, nd, dec_tables.shape[1]))
    side, main = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1)
    side.wait_stream(torch.cuda.current_stream())
    main.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        batch.launch(stream=side)
    for l in range(nl):
        zipage.zp_paged_decode_attn(batch.pool, l, inp.decode_q[l], dec_tables, dec_seq, outs[l], p, ws, stream=main)
    torch.cuda.synchronize()
    assert batch.error(side) == 0
    assert zipage.zp_read_error(ws, main) == 0
    # compression: every unit's compaction, then sampled units against the oracle
    _compaction_property_all_units(batch, pristine, batch.debug["keep"])
    check_sampled_units(batch, inp, pristine, gs_in, seed=5)
    # decode: the decode requests' blocks are disjoint from the compressing ones
    got = outs.float().cpu().numpy()
    qb = synth.bf16_bits(inp.decode_q.cpu())
    G = wl.num_q_heads // wl.num_kv_heads
    b = wl.block_size
    dseq = inp.seq_len[R:]
    rng = np.random.default_rng(9)
    picks = {(0, int(np.argmin(dseq))), (nl - 1, int(np.argmax(dseq)))}
    picks |= {(int(rng.integers(nl)), int(rng.integers(nd))) for _ in range(10)}
    for l, i in sorted(picks):
        s = int(dseq[i])
        tab = torch.from_numpy(inp.block_tables[R + i]).long().cuda()
        t = torch.arange(s, device="cuda")
        for h in range(wl.num_kv_heads):
            k = synth.bf16_bits(pristine[l, tab[t // b], 0, h, t % b])
            v = synth.bf16_bits(pristine[l, tab[t // b], 1, h, t % b])
            want = O.decode_attention(qb[l, i, h * G:(h + 1) * G], k, v, wl.scale)
            err = np.abs(got[l, i, h * G:(h + 1) * G] - want)
            assert (err <= DEC_RTOL * np.abs(want) + DEC_ATOL).all(), (l, i, h, float(err.max()))
    batch.close()
