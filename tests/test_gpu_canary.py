"""Out-of-bounds write checks (a stand-in for a memory sanitiser): every workspace is followed by
a canary band that no call may touch, and the slots of the global scores and of the per-token
outputs past each request's length stay as they were."""
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


@pytest.mark.parametrize("name,wl", [
    ("prefill_small", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=2, n_max=32, prefill_max=1100)),
    ("long_prefill", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                                       n_max=64, prefill_max=4000)),
    ("multipass", synth.WORKLOADS["prefill"].scaled(num_requests=4, num_layers=1, num_kv_heads=2, num_q_heads=8,
                                                    n_max=64, prefill_max=9000)),
])
def test_compress_writes_stay_in_bounds(zp, name, wl):
    zipage, runner = zp
    inp = synth.make_inputs(wl, "cpu")
    batch = runner.CompressionBatch(inp, "cuda")
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
    gs_after = batch.gs.cpu().numpy()
    gsb = gs_before.cpu().numpy()
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
    out = torch.zeros_like(q)
    ws, band = _banded(zipage.zp_paged_decode_workspace_size(p, B, mb))
    zipage.zp_paged_decode_attn(pool, 1, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == 0
    torch.cuda.synchronize()
    assert bool((band == CANARY).all()), "decode wrote past its workspace"
    red = torch.full((B, layers, Hkv, mb * b), -7.0, device="cuda")
    ws, band = _banded(zipage.zp_redundancy_workspace_size(p, B))
    zipage.zp_redundancy_all_pairs(pool, tables, seq, red, p, ws)
    assert zipage.zp_read_error(ws) == 0
    torch.cuda.synchronize()
    assert bool((band == CANARY).all()), "all-pairs redundancy wrote past its workspace"
    assert torch.isfinite(red).all()
