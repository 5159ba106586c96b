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

# the tolerance of the decode tests: bf16 output rounding (2^-9 relative) plus fp32 accumulation
RTOL, ATOL = 4e-3, 1e-4


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


def _with_workspace(zipage, pool, tables, q, seq, p, layer):
    out = torch.zeros_like(q)
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, q.shape[0], tables.shape[1]))
    zipage.zp_paged_decode_attn(pool, layer, q, tables, seq, out, p, ws)
    assert zipage.zp_read_error(ws) == 0
    return out.float()


def test_static_scratch_matches_workspace_variant_twice(zipage):
    # call 1 spans several splits per request; call 2 is smaller, so partials left in the
    # shared array by call 1 would show up if they leaked into call 2
    cases = [_case(11, [1, 17, 300, 1100, 2048, 513], layers=2), _case(12, [40, 16, 257], layers=3)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for (pool, tables, q, seq, p), layer in zip(cases, (1, 2)):
        want = _with_workspace(zipage, pool, tables, q, seq, p, layer)
        out = torch.zeros_like(q)
        zipage.zp_paged_decode_attn_static(pool, layer, q, tables, seq, out, p, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.float()
        assert torch.all((got - want).abs() <= RTOL * want.abs() + ATOL)


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
