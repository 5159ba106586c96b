"""The hybrid scheduler driving the CUDA kernels for a few hundred engine steps on a seeded
synthetic trace (no model: new tokens get random keys and values, window queries are random).
The scheduler's compressions (decode-trigger and prefill-overshoot ones) run through
zp_compress on a side stream and its decoding requests through zp_paged_decode_attn on the main
stream (serialised here, so that the first compressions can be checked against the oracle on
exact pool contents); the scheduler releases the blocks past N_max-1 when it applies a
compression.  Every request finishes."""
import numpy as np
import pytest
import torch

from oracle import parity
from paged_kv_cache_obs_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zp():
    import os
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage
    return zipage


def test_scheduler_drives_compression_and_decode(zp):
    layers, Hq, Hkv, d, b, n_max, w, M = 2, 8, 2, 64, 16, 6, 8, 3
    NB = 160
    g = torch.Generator(device="cuda").manual_seed(11)
    pool = torch.randn((layers, NB, 2, Hkv, b, d), generator=g, device="cuda").to(torch.bfloat16)
    p = dict(num_layers=layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=b, n_max=n_max,
             window=w, alpha=0.5, beta=0.5, decay=0.9, scale=1.0 / np.sqrt(d), protect_window=1, causal=1)
    alloc = zp.zp_alloc_create(NB)
    sched = zp.zp_sched_create(alloc, n_max, b, M)
    rng = np.random.default_rng(3)
    ids = [zp.zp_sched_submit(sched, int(rng.integers(10, 150)), int(rng.integers(20, 200))) for _ in range(10)]
    L_max = 150 + 16   # longest prompt rounded up: the global-score row length
    gs = torch.zeros((M, layers, Hkv, L_max), device="cuda")
    slot_of = {}
    side, main = torch.cuda.Stream(), torch.cuda.current_stream()
    ws_c = zp.new_workspace(zp.zp_compress_workspace_size(p, len(ids)))
    checked = 0
    try:
        for step in range(400):
            plan = zp.zp_sched_step(sched)
            infos = {i: zp.zp_sched_request(sched, i) for i in ids}
            if all(infos[i]["state"] == 2 for i in ids):
                break
            # query slots of this step (the scheduler decides who holds one)
            holders = [i for i in ids if infos[i]["state"] == 1 and infos[i]["has_slot"]]
            for i in list(slot_of):
                if i not in holders:
                    del slot_of[i]
            for i in holders:
                if i not in slot_of:
                    slot_of[i] = min(set(range(M)) - set(slot_of.values()))
            comp = plan["compress"]
            if comp:
                R = len(comp)
                mb = max(max(infos[i]["num_blocks"] for i in comp), -(-L_max // b))
                tables = np.full((R, mb), -1, np.int32)
                for r, i in enumerate(comp):
                    tables[r, :infos[i]["num_blocks"]] = infos[i]["table"]
                seq = np.array([infos[i]["seq_len"] for i in comp], np.int32)
                qs = np.array([slot_of[i] for i in comp], np.int32)
                obs_q = torch.randn((M, layers, w, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
                pool_in = synth.bf16_bits(pool) if checked < 3 else None
                gs_in = gs.cpu().numpy() if checked < 3 else None
                dbg = {k: torch.zeros((R, layers, Hkv, L_max), device="cuda", dtype=dt)
                       for k, dt in (("attn", torch.float32), ("redund", torch.float32),
                                     ("score", torch.float32), ("keep", torch.int32))}
                side.wait_stream(main)
                with torch.cuda.stream(side):
                    dt_ = torch.from_numpy(tables).to("cuda", non_blocking=False)
                    zp.zp_compress(pool, dt_, torch.from_numpy(seq).cuda(), torch.from_numpy(qs).cuda(), dt_, obs_q,
                                   gs, p, ws_c, debug=dbg, stream=side, max_seq_len=L_max)
                side.synchronize()
                assert zp.zp_read_error(ws_c, side) == 0
                if checked < 3:
                    units = [(r, l, h) for r in range(R) for l in range(layers) for h in range(Hkv)]
                    parity.check_units(units, pool_in, synth.bf16_bits(obs_q), gs_in, tables, tables, seq, qs, p,
                                       {k: v.cpu().numpy() for k, v in dbg.items()}, gs.cpu().numpy(),
                                       synth.bf16_bits(pool), full_pool=True)
                    checked += 1
            dec = plan["decode"]
            if dec:
                # append the new token's K/V (random) at position seq_len, then decode over it
                for i in dec:
                    inf = infos[i]
                    pos = inf["seq_len"]
                    blk = inf["table"][pos // b]
                    pool[:, blk, :, :, pos % b] = torch.randn((layers, 2, Hkv, d), generator=g,
                                                              device="cuda").to(torch.bfloat16)
                B = len(dec)
                mb = max(infos[i]["num_blocks"] for i in dec)
                tables = np.full((B, mb), -1, np.int32)
                for r, i in enumerate(dec):
                    tables[r, :infos[i]["num_blocks"]] = infos[i]["table"]
                seq = torch.tensor([infos[i]["seq_len"] + 1 for i in dec], dtype=torch.int32, device="cuda")
                q = torch.randn((B, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
                out = torch.empty_like(q)
                ws = zp.new_workspace(zp.zp_paged_decode_workspace_size(p, B, mb))
                for l in range(layers):
                    zp.zp_paged_decode_attn(pool, l, q, torch.from_numpy(tables).cuda(), seq, out, p, ws)
                assert zp.zp_read_error(ws) == 0
                assert torch.isfinite(out.float()).all()
        st = zp.zp_sched_get_stats(sched)
        assert st["finished"] == len(ids)
        assert st["compressions"] >= 3 and checked >= 3
    finally:
        zp.zp_sched_destroy(sched)
        zp.zp_alloc_destroy(alloc)
