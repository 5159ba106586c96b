"""Out-of-bounds write checks (a stand-in for a memory sanitiser): every workspace is followed by
a canary band, and the KV pool, the global scores and the outputs lie between two bands, that
no call may touch; the global scores of idle query slots and the slots of the global scores and
of the per-token outputs past each request's length stay as they were, and calls that only read
the pool leave it unchanged."""
import numpy as np
import pytest
import torch

from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu

CANARY = 0xA5
BAND = 4096


@pytest.fixture(scope="module")
def zp():
    import os
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import runner, zipage
    return zipage, runner


def _banded(nbytes):
    """A device buffer of nbytes (rounded up to 256) followed by a canary band; returns (view, band)."""
    n = (nbytes + 255) // 256 * 256
    buf = torch.full((n + BAND,), CANARY, dtype=torch.uint8, device="cuda")
    return buf[:n], buf[n:]


def _fenced_copy(t):
    """A device copy of tensor t between two canary bands; returns (copy, bands).  The copy
    starts 256-byte aligned, as every buffer the library takes must be 16-byte aligned."""
    nbytes = t.numel() * t.element_size()
    n = (nbytes + 255) // 256 * 256
    buf = torch.full((BAND + n + BAND,), CANARY, dtype=torch.uint8, device="cuda")
    view = buf[BAND:BAND + nbytes].view(t.dtype).view(t.shape)
    view.copy_(t.to("cuda"))
    return view, (buf[:BAND], buf[BAND + n:])


def _intact(bands):
    return all(bool((b == CANARY).all()) for b in bands)


@pytest.mark.parametrize("name,wl", [
    ("trigger", synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2)),
    ("prefix", synth.WORKLOADS["shared_prefix"].scaled(num_requests=3, num_layers=1, num_kv_heads=2, num_q_heads=8)),
    ("prefill_small", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=2, n_max=32, prefill_max=1100)),
    ("long_prefill", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                                       n_max=64, prefill_max=4000)),
    ("multipass", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                                    n_max=64, prefill_max=9000)),
])
def test_compress_writes_stay_in_bounds(zp, name, wl):
    zipage, runner = zp
    inp = synth.make_inputs(wl, "cpu")
    pool, pool_bands = _fenced_copy(inp.pool)  # the KV pool and the global scores between bands
    batch = runner.CompressionBatch(inp, "cuda", pool=pool)
    batch.gs, gs_bands = _fenced_copy(inp.global_scores)
    batch.enable_debug()
    for v in batch.debug.values():
        v.fill_(-7)
    R = inp.num_compress
    need = zipage.zp_compress_workspace_size(batch.params, R, batch.max_seq_len)
    batch.workspace, band = _banded(need)
    gs_before = batch.gs.clone()
    batch.launch()
    assert batch.error() == 0
    torch.cuda.synchronize()
    assert bool((band == CANARY).all()), "a write past the workspace"
    assert _intact(pool_bands), "a write outside the KV pool"
    assert _intact(gs_bands), "a write outside the global scores"
    gs_after = batch.gs.cpu().numpy()
    gsb = gs_before.cpu().numpy()
    # the query slots of no compressing request keep their global scores
    idle = sorted(set(range(gsb.shape[0])) - {int(x) for x in inp.qslot[:R]})
    assert np.array_equal(gs_after[idle], gsb[idle]), "global scores of an idle query slot"
    dbg = {k: v.cpu().numpy() for k, v in batch.debug.items()}
    for r in range(R):
        L, s = int(inp.seq_len[r]), int(inp.qslot[r])
        assert np.array_equal(gs_after[s, :, :, L:], gsb[s, :, :, L:]), (r, "global scores past L")
        for k, v in dbg.items():
            assert (v[r, :, :, L:] == -7).all(), (r, k, "per-token output past L")
    batch.close()


def test_decode_and_all_pairs_workspaces_stay_in_bounds(zp):
    zipage, _ = zp
    g = torch.Generator().manual_seed(3)
    layers, Hq, Hkv, d, b = 2, 8, 2, 128, 16
    seq_lens = [1, 15, 300, 777]
    B = len(seq_lens)
    mb = max((s + b - 1) // b for s in seq_lens)
    NB = B * mb + 3
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g).to(torch.bfloat16).cuda()
    tables = torch.from_numpy(torch.randperm(NB, generator=g).numpy()[:B * mb].reshape(B, mb).astype(np.int32)).cuda()
    seq = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    p = dict(num_layers=layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=mb,
             window=1, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16).cuda()
    out, out_bands = _fenced_copy(torch.zeros((B, Hq, d), dtype=torch.bfloat16))
    pool_in = pool.clone()
    ws, band = _banded(zipage.zp_paged_decode_workspace_size(p, B, mb))
    zipage.zp_paged_decode_attn(pool, 1, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == 0
    torch.cuda.synchronize()
    assert bool((band == CANARY).all()), "decode wrote past its workspace"
    assert _intact(out_bands), "decode wrote outside its output"
    red, red_bands = _fenced_copy(torch.full((B, layers, Hkv, mb * b), -7.0))
    ws, band = _banded(zipage.zp_redundancy_workspace_size(p, B))
    zipage.zp_redundancy_all_pairs(pool, tables, seq, red, p, ws)
    assert zipage.zp_read_error(ws) == 0
    torch.cuda.synchronize()
    assert bool((band == CANARY).all()), "all-pairs redundancy wrote past its workspace"
    assert _intact(red_bands), "all-pairs redundancy wrote outside its output"
    assert torch.isfinite(red).all()
    assert torch.equal(pool.view(torch.int16), pool_in.view(torch.int16)), "a read-only call wrote to the pool"
