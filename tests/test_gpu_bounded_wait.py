"""Failure detection by bounded waits, exercised without a GPU fault.

Every wait inside the kernels is bounded; a wait that runs out makes the kernel finish its
in-flight copies, record ZP_ERR_TIMEOUT in the error word and return, so the context stays
usable.  zp_test_decode_stalled and zp_test_compress_stalled make the decode kernel and the
multi-pass compression's statistics kernel wait, briefly, on a barrier that nothing ever
completes, so that this path runs for real: the tests check the reported status, that no write
leaves its buffer, and that the next ordinary call on the same context is correct."""
import numpy as np
import pytest
import torch

from oracle import parity
from oracle import zipage_oracle as O
from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu

CANARY = 0xA5
BAND = 4096
DEC_RTOL, DEC_ATOL = 4e-3, 1e-4


@pytest.fixture(scope="module")
def zipage():
    import os
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage as z
    return z


def _banded(nbytes, dtype=torch.uint8):
    n = (nbytes + 255) // 256 * 256
    buf = torch.full((n + BAND,), CANARY, dtype=torch.uint8, device="cuda")
    return buf[:n], buf[n:]


def test_decode_wait_that_runs_out_reports_timeout_and_context_survives(zipage):
    g = torch.Generator().manual_seed(21)
    layers, Hq, Hkv, d, b = 2, 8, 2, 128, 16
    seq_lens = [5, 300, 1100, 2048]              # one to several splits per request
    B = len(seq_lens)
    mb = max((s + b - 1) // b for s in seq_lens)
    NB = B * mb + 3
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g).to(torch.bfloat16).cuda()
    tables = torch.from_numpy(torch.randperm(NB, generator=g).numpy()[:B * mb].reshape(B, mb).astype(np.int32)).cuda()
    seq = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16).cuda()
    p = dict(num_layers=layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=mb,
             window=1, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    # output and workspace, each followed by a canary band
    obuf, oband = _banded(B * Hq * d * 2)
    out = obuf.view(torch.bfloat16)[:B * Hq * d].view(B, Hq, d)
    ws, wband = _banded(zipage.zp_paged_decode_workspace_size(p, B, mb))
    pool_before = pool.clone()

    zipage.zp_test_decode_stalled(pool, 1, q, tables, seq, out, p, ws, stall_limit_ns=2_000_000)
    assert zipage.zp_read_error(ws) == zipage.ZP_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert bool((oband == CANARY).all()) and bool((wband == CANARY).all())
    assert torch.equal(pool.view(torch.int16), pool_before.view(torch.int16))
    # no key was folded in before the wait gave up: every output is the empty sum
    assert not out.float().any()

    # the context is intact: an ordinary call on it matches the oracle
    zipage.zp_paged_decode_attn(pool, 1, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == 0
    torch.cuda.synchronize()
    assert bool((oband == CANARY).all()) and bool((wband == CANARY).all())
    got = O.bf16_bits_to_f64(synth.bf16_bits(out))
    pb, qb = synth.bf16_bits(pool), synth.bf16_bits(q)
    tb = tables.cpu().numpy()
    G = Hq // Hkv
    for r, s in enumerate(seq_lens):
        for h in range(Hkv):
            k = O.gather_rows(pb, 1, 0, h, tb[r], s, b)
            v = O.gather_rows(pb, 1, 1, h, tb[r], s, b)
            want = O.decode_attention(qb[r, h * G:(h + 1) * G], k, v, p["scale"])
            err = np.abs(got[r, h * G:(h + 1) * G] - want)
            assert (err <= DEC_RTOL * np.abs(want) + DEC_ATOL).all(), (r, h)


def test_stall_limit_is_validated(zipage):
    pool = torch.zeros((1, 4, 2, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    tables = torch.arange(4, dtype=torch.int32, device="cuda").view(1, 4)
    seq = torch.tensor([20], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    p = dict(num_layers=1, num_q_heads=1, num_kv_heads=1, head_dim=64, block_size=16, n_max=4, window=1,
             alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, 1, 4))
    for bad in (0, -5, 2_000_000_000):
        with pytest.raises(zipage.ZipageError) as e:
            zipage.zp_test_decode_stalled(pool, 0, q, tables, seq, out, p, ws, stall_limit_ns=bad)
        assert e.value.status == zipage.ZP_ERR_INVALID_ARG


def test_compression_wait_that_runs_out_reports_timeout_and_context_survives(zipage):
    # the multi-pass form (a launch length above 4096): its CTAs exchange nothing, so a wait that
    # gives up stays inside its CTA
    from paged_kv_cache_obs_gb300 import runner
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=2, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                           n_max=64, prefill_max=5000)
    inp = synth.make_inputs(wl, "cpu")
    R = inp.num_compress
    pool_in = synth.bf16_bits(inp.pool)
    gs_in = inp.global_scores.numpy().copy()
    obs_q = synth.bf16_bits(inp.obs_q)
    batch = runner.CompressionBatch(inp, "cuda")
    assert batch.max_seq_len > 4096
    pristine, gs0 = batch.pool.clone(), batch.gs.clone()
    ws, wband = _banded(zipage.zp_compress_workspace_size(batch.params, R, batch.max_seq_len))
    with pytest.raises(zipage.ZipageError):  # only the multi-pass form takes the hook
        zipage.zp_test_compress_stalled(batch.pool, batch.d_tables, batch.d_seq, batch.d_qslot, batch.d_dst,
                                        batch.obs_q, batch.gs, batch.params, ws, stall_limit_ns=2_000_000,
                                        max_seq_len=4096)
    zipage.zp_test_compress_stalled(batch.pool, batch.d_tables, batch.d_seq, batch.d_qslot, batch.d_dst,
                                    batch.obs_q, batch.gs, batch.params, ws, stall_limit_ns=2_000_000,
                                    max_seq_len=batch.max_seq_len)
    assert zipage.zp_read_error(ws) == zipage.ZP_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert bool((wband == CANARY).all())
    # blocks outside every table of the call are untouched
    used = set(batch.tables.ravel().tolist()) | set(batch.dst_tables.ravel().tolist())
    others = [blk for blk in range(inp.pool.shape[1]) if blk not in used]
    assert torch.equal(batch.pool[:, others].view(torch.int16), pristine[:, others].view(torch.int16))

    # the context is intact: the ordinary call on the restored inputs matches the oracle
    batch.pool.copy_(pristine)
    batch.gs.copy_(gs0)
    batch.workspace = ws
    batch.enable_debug()
    batch.launch()
    assert batch.error() == 0
    torch.cuda.synchronize()
    assert bool((wband == CANARY).all())
    units = [(r, l, h) for r in range(R) for l in range(wl.num_layers) for h in range(wl.num_kv_heads)]
    dbg = {k: v.cpu().numpy() for k, v in batch.debug.items()}
    ndiff = parity.check_units(units, pool_in, obs_q, gs_in, batch.tables, batch.dst_tables, inp.seq_len[:R],
                               inp.qslot, wl.params(), dbg, batch.gs.cpu().numpy(), synth.bf16_bits(batch.pool),
                               full_pool=True, n_max_per_req=inp.n_max_req)
    assert ndiff <= 2
    batch.close()
