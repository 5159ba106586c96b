"""zp_paged_decode_attn_static: decode attention for callers that cannot allocate device
memory (a host runtime that owns all device buffers through its own pool, a serving loop that
must not call cudaMalloc in its hot path, a process whose device footprint must be fixed when
the library loads).  Its scratch is the library's fixed device array, so no workspace is
passed; its results must equal those of zp_paged_decode_attn, call after call.

Collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test."""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zipage():
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage as z
    return z


def _case(seed, seq_lens, Hq=32, Hkv=8, d=128, b=16, layers=2):
    g = torch.Generator().manual_seed(seed)
    B = len(seq_lens)
    max_blocks = max((s + b - 1) // b for s in seq_lens) + 2
    NB = B * max_blocks + 5
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g).to(torch.bfloat16).cuda()
    tables = torch.randperm(NB, generator=g)[:B * max_blocks].view(B, max_blocks).to(torch.int32).cuda()
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16).cuda()
    seq = torch.tensor(seq_lens, dtype=torch.int32).cuda()
    p = dict(num_layers=layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=max_blocks,
             window=1, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    return pool, tables, q, seq, p


def _with_workspace(zipage, pool, tables, q, seq, p, layer, expect=0):
    out = torch.zeros_like(q)
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, q.shape[0], tables.shape[1]))
    zipage.zp_paged_decode_attn(pool, layer, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == expect
    return out


def test_static_scratch_matches_workspace_variant_twice(zipage):
    # Both entry points run the same kernels with the same split size and differ only in where
    # the split partials live, so the outputs must be bit-identical.  Call 1 spans several
    # splits per request; call 2 is smaller, so partials left in the shared array by call 1
    # would show up if they leaked into call 2.
    cases = [_case(11, [1, 17, 300, 1100, 2048, 513], layers=2), _case(12, [40, 16, 257], layers=3)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for (pool, tables, q, seq, p), layer in zip(cases, (1, 2)):
        want = _with_workspace(zipage, pool, tables, q, seq, p, layer)
        out = torch.zeros_like(q)
        zipage.zp_paged_decode_attn_static(pool, layer, q, tables, seq, out, p, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, want)


def test_static_scratch_reports_a_bad_request_then_recovers(zipage):
    # A request whose length exceeds its table is reported through dev_status and left alone;
    # the other requests are still computed.  The next call, with no status word (device-side
    # errors go to the array's spare word), starts from a clean state and matches again.
    pool, tables, q, seq, p = _case(14, [300, 1100, 700, 64], layers=2)
    max_blocks = tables.shape[1]
    bad = seq.clone()
    bad[1] = max_blocks * p["block_size"] + 1
    want = _with_workspace(zipage, pool, tables, q, bad, p, 1, expect=zipage.ZP_ERR_BAD_TABLE)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    sentinel = torch.full_like(q, 7.0)
    out = sentinel.clone()
    zipage.zp_paged_decode_attn_static(pool, 1, q, tables, bad, out, p, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == zipage.ZP_ERR_BAD_TABLE
    good = [0, 2, 3]
    assert torch.equal(out[good], want[good])
    assert torch.equal(out[1], sentinel[1])          # the bad request's output is untouched
    want2 = _with_workspace(zipage, pool, tables, q, seq, p, 0)
    out2 = torch.zeros_like(q)
    zipage.zp_paged_decode_attn_static(pool, 0, q, tables, seq, out2, p, dev_status=None)
    torch.cuda.synchronize()
    assert torch.equal(out2, want2)


def test_static_scratch_rejects_calls_beyond_its_size(zipage):
    pool, tables, q, seq, p = _case(13, [64, 64])
    big_q = q.repeat(4000, 1, 1)                      # 8000 requests x 32 heads: far beyond 16 MiB
    big_t = tables.repeat(4000, 1)
    big_s = seq.repeat(4000)
    out = torch.zeros_like(big_q)
    with pytest.raises(zipage.ZipageError) as e:
        zipage.zp_paged_decode_attn_static(pool, 0, big_q, big_t, big_s, out, p)
    assert e.value.status == zipage.ZP_ERR_TOO_LARGE
    assert not out.any()
