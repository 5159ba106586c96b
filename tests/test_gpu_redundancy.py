"""GPU parity of the original all-pairs redundancy (zp_redundancy_all_pairs), the ablation of
the Lightning Redundancy Score, against the fp64 oracle.

Tolerance.  The kernel forms each Gram entry on the tensor cores from exact bf16 products with
fp32 accumulation over d <= 128 terms (relative error below d * 2^-24 ~ 8e-6 of |k_t||k_j|, so
below 8e-6 in cosine units), takes the norms from an fp32 sum of squares (~1e-6), and averages
L - 1 such cosines in fp32.  The mean is therefore within ~1e-5 of the exact value; the test
allows 5e-5 absolute plus 1e-4 relative."""
import numpy as np
import pytest
import torch

from oracle import zipage_oracle as O
from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 5e-5, 1e-4


@pytest.fixture(scope="module")
def zp():
    import os
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage
    return zipage


def _case(zipage, *, layers, Hkv, d, b, seq_lens, L_max=0, seed=0, heavy=False):
    g = torch.Generator().manual_seed(seed)
    R = len(seq_lens)
    L_row = L_max or max(seq_lens)
    mb = (L_row + b - 1) // b
    NB = R * mb + 5
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g)
    if heavy:  # a few directions shared by many keys, and some large keys: high redundancy
        cent = torch.randn((4, d), generator=g)
        idx = torch.randint(0, 4, (layers, NB, Hkv, b), generator=g)
        pool[:, :, 0] = cent[idx] * 3 + 0.1 * pool[:, :, 0]
    pool = pool.to(torch.bfloat16)
    perm = torch.randperm(NB, generator=g).numpy().astype(np.int32)
    tables = perm[:R * mb].reshape(R, mb).copy()
    p = dict(num_layers=layers, num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=mb,
             window=1, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    out = torch.full((R, layers, Hkv, L_row), float("nan"), device="cuda")
    ws = zipage.new_workspace(zipage.zp_redundancy_workspace_size(p, R, L_row))
    zipage.zp_redundancy_all_pairs(pool.cuda(), torch.from_numpy(tables).cuda(),
                                   torch.tensor(seq_lens, dtype=torch.int32).cuda(), out, p, ws,
                                   max_seq_len=L_row)
    assert zipage.zp_read_error(ws) == 0
    got = out.cpu().numpy()
    pb = synth.bf16_bits(pool)
    for r, L in enumerate(seq_lens):
        for l in range(layers):
            for h in range(Hkv):
                k = O.bf16_bits_to_f64(O.gather_rows(pb, l, 0, h, tables[r], L, b))
                want = O.all_pairs_redundancy(k)
                err = np.abs(got[r, l, h, :L] - want)
                assert (err <= ATOL + RTOL * np.abs(want)).all(), (r, l, h, float(err.max()))
                assert (got[r, l, h, L:] == 0).all()
    return got


@pytest.mark.parametrize("d,b", [(128, 16), (128, 32), (64, 16), (64, 32)])
def test_all_pairs_ragged_lengths(zp, d, b):
    # one tile, a ragged tile, a partial block, several tiles, L = 1 and L = 2
    _case(zp, layers=2, Hkv=2, d=d, b=b, seq_lens=[100, 128, 129, 300, 1, 2, 383], seed=d + b)


def test_all_pairs_high_redundancy(zp):
    got = _case(zp, layers=1, Hkv=2, d=128, b=16, seq_lens=[640, 257], seed=5, heavy=True)
    assert got[0, 0, 0, :640].mean() > 0.2  # the clustered keys are redundant


def test_all_pairs_full_length_sample(zp):
    # the Llama-3-8B workload's length (N_max = 128 blocks of 16) on a few units
    _case(zp, layers=2, Hkv=2, d=128, b=16, seq_lens=[2048, 2048, 1999], seed=9)


def test_all_pairs_bad_block_reports(zp):
    p = dict(num_layers=1, num_q_heads=2, num_kv_heads=2, head_dim=64, block_size=16, n_max=4, window=1,
             alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    pool = torch.zeros((1, 8, 2, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    tables = torch.tensor([[0, 1, 99, 2]], dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 1, 2, 64), device="cuda")
    ws = zp.new_workspace(zp.zp_redundancy_workspace_size(p, 1))
    zp.zp_redundancy_all_pairs(pool, tables, torch.tensor([50], dtype=torch.int32, device="cuda"), out, p, ws)
    assert zp.zp_read_error(ws) == zp.ZP_ERR_BAD_TABLE
