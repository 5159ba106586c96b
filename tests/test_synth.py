"""The seeded input generators: the same seed gives the same bytes (both sides of every parity
test read them), another seed gives other bytes, and the workloads have the shapes and
structure their recipes state."""
import numpy as np
import torch

from paged_kv_cache_obs_gb300 import synth


def _bytes(inp):
    return (synth.bf16_bits(inp.pool), synth.bf16_bits(inp.obs_q), inp.global_scores.numpy(),
            inp.block_tables, inp.seq_len, inp.qslot)


def test_same_seed_same_bytes():
    wl = synth.WORKLOADS["llama3_8b"].scaled(num_requests=2, num_layers=2)
    a, b = _bytes(synth.make_inputs(wl, "cpu")), _bytes(synth.make_inputs(wl, "cpu"))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    c = _bytes(synth.make_inputs(wl, "cpu", seed=synth.seed_of(wl) + 1))
    assert not np.array_equal(a[0], c[0])


def test_workload_structure():
    # prefill overshoot: every request holds more than k tokens and at most prefill_max
    wl = synth.WORKLOADS["prefill"].scaled(num_requests=6, num_layers=1)
    inp = synth.make_inputs(wl, "cpu")
    k = (wl.n_max - 1) * wl.block_size
    assert ((inp.seq_len[:6] > k) & (inp.seq_len[:6] <= wl.prefill_max)).all()
    # shared prefix: the first 16 blocks are the same physical blocks in every request
    wl = synth.WORKLOADS["shared_prefix"].scaled(num_requests=3, num_layers=1)
    inp = synth.make_inputs(wl, "cpu")
    t = inp.block_tables[:3, :16]
    assert (t == t[0]).all()
    assert (inp.refcount[t[0]] == 3 + 1).all()
    # block ids of different requests are otherwise disjoint
    own = [set(inp.block_tables[r, 16:wl.n_max].tolist()) for r in range(3)]
    assert not (own[0] & own[1]) and not (own[1] & own[2])


def test_large_requested_pool_draws_the_referenced_blocks():
    # the mixed workload's pool is far larger than the blocks in use: only the blocks of some
    # table are drawn, with the same recipe, and the ids spread over the whole pool
    wl = synth.WORKLOADS["mixed"].scaled(num_requests=2, num_layers=2, num_decode=3, pool_blocks=4000)
    inp = synth.make_inputs(wl, "cpu")
    assert inp.pool.shape[1] == 4000
    used = np.unique(inp.block_tables[inp.block_tables >= 0])
    assert (inp.refcount[used] >= 1).all()
    assert used.max() > 1000  # a permutation of the whole pool, not of its first blocks
    k = inp.pool[:, torch.as_tensor(used), 0].float()
    v = inp.pool[:, torch.as_tensor(used), 1].float()
    assert torch.isfinite(k).all() and torch.isfinite(v).all()
    assert float(v.std()) > 0.5 and float(k.abs().mean()) > 0.1
