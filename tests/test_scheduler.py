"""Hybrid scheduler of Compressed PagedAttention (host, no GPU): the policy of the pages' hybrid
scheduling (query slots for the first M running requests, slot-less decoding below the block
cap, compression only with a slot, preemption of slot-less requests first, restricted mode),
checked step by step on seeded synthetic request traces."""
import os

import numpy as np
import pytest


@pytest.fixture(scope="module")
def zp():
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage
    return zipage


def _run(zp, prompts, gens, pool, n_max, b, M, max_steps=100000, check=True):
    a = zp.zp_alloc_create(pool)
    s = zp.zp_sched_create(a, n_max, b, M)
    ids = [zp.zp_sched_submit(s, int(p), int(g)) for p, g in zip(prompts, gens)]
    running_hist = []
    steps = 0
    try:
        while True:
            plan = zp.zp_sched_step(s)
            steps += 1
            infos = {i: zp.zp_sched_request(s, i) for i in ids}
            running = [i for i in ids if infos[i]["state"] == 1]
            running_hist.append(len(running))
            if check:
                held = sum(infos[i]["num_blocks"] for i in running)
                assert held + zp.zp_num_free(a) == pool                     # every block accounted for
                assert sum(infos[i]["has_slot"] for i in running) <= M      # at most M slots
                for i in running:
                    inf = infos[i]
                    blocks_needed = -(-inf["seq_len"] // b)
                    assert inf["num_blocks"] in (blocks_needed, blocks_needed + 1)
                    if inf["num_blocks"] > n_max:                           # only a prefill overshoot
                        assert inf["seq_len"] > n_max * b or i in plan["prefill"]
                for i in plan["compress"]:
                    assert infos[i]["has_slot"]                            # compression needs a slot
                assert not set(plan["compress"]) & set(plan["decode"])
                for i in plan["preempted"]:
                    assert infos[i]["state"] == 0 and not infos[i]["has_slot"]
                    assert infos[i]["num_blocks"] == 0
            if all(infos[i]["state"] == 2 for i in ids):
                break
            assert steps < max_steps, "no progress"
        return zp.zp_sched_get_stats(s), running_hist, steps
    finally:
        zp.zp_sched_destroy(s)
        zp.zp_alloc_destroy(a)


def test_random_trace_invariants_and_completion(zp):
    rng = np.random.default_rng(0)
    n = 60
    prompts = rng.integers(8, 600, size=n)
    gens = rng.integers(1, 1200, size=n)
    stats, hist, steps = _run(zp, prompts, gens, pool=220, n_max=16, b=16, M=6)
    assert stats["finished"] == n
    assert stats["decoded_tokens"] >= gens.sum()          # preempted work is recomputed
    assert stats["compressions"] > 0


def test_slots_go_to_the_earliest_running_requests(zp):
    a = zp.zp_alloc_create(400)
    s = zp.zp_sched_create(a, 8, 16, 2)
    try:
        ids = [zp.zp_sched_submit(s, 20, 500) for _ in range(5)]
        zp.zp_sched_step(s)
        slots = [zp.zp_sched_request(s, i)["has_slot"] for i in ids]
        assert slots == [True, True, False, False, False]
        # slot-less requests still decode (hybrid scheduling: concurrency above M)
        plan = zp.zp_sched_step(s)
        assert sorted(plan["decode"]) == ids
    finally:
        zp.zp_sched_destroy(s)
        zp.zp_alloc_destroy(a)


def test_compression_needs_a_slot_and_keeps_the_cap(zp):
    b, n_max = 16, 4
    a = zp.zp_alloc_create(100)
    s = zp.zp_sched_create(a, n_max, b, 1)
    try:
        r0 = zp.zp_sched_submit(s, n_max * b, 100)   # holds the slot, at the cap at once
        r1 = zp.zp_sched_submit(s, n_max * b, 100)   # no slot, at the cap
        plan = zp.zp_sched_step(s)
        assert plan["compress"] == [r0] and r1 not in plan["decode"]
        plan = zp.zp_sched_step(s)                   # r0's compression applied: k tokens
        info = zp.zp_sched_request(s, r0)
        assert info["seq_len"] == (n_max - 1) * b          # decoded tokens land at the next step
        assert r0 in plan["decode"]
        assert info["num_blocks"] <= n_max
        assert zp.zp_sched_get_stats(s)["slot_waits"] >= 2
    finally:
        zp.zp_sched_destroy(s)
        zp.zp_alloc_destroy(a)


def test_prefill_longer_than_the_cap_is_compressed_first(zp):
    b, n_max = 16, 4
    a = zp.zp_alloc_create(64)
    s = zp.zp_sched_create(a, n_max, b, 2)
    try:
        r = zp.zp_sched_submit(s, 150, 10)            # 10 blocks > n_max: prefill overshoot
        plan = zp.zp_sched_step(s)
        assert plan["prefill"] == [r] and plan["compress"] == [r]
        zp.zp_sched_step(s)
        info = zp.zp_sched_request(s, r)
        assert info["num_blocks"] <= n_max and info["seq_len"] <= n_max * b
    finally:
        zp.zp_sched_destroy(s)
        zp.zp_alloc_destroy(a)


def test_preemption_takes_the_latest_slotless_request_first(zp):
    b = 16
    a = zp.zp_alloc_create(10)
    s = zp.zp_sched_create(a, 8, b, 1)
    try:
        ids = [zp.zp_sched_submit(s, 2 * b, 400) for _ in range(5)]   # 5 x 2 blocks = the pool
        preempted = []
        for _ in range(40):
            plan = zp.zp_sched_step(s)
            preempted += plan["preempted"]
            if preempted:
                break
        assert preempted[:2] == [ids[4], ids[3]]                     # newest slot-less first
        assert ids[0] not in preempted                               # the slot holder survives
    finally:
        zp.zp_sched_destroy(s)
        zp.zp_alloc_destroy(a)


def test_compression_raises_concurrency_on_a_fixed_pool(zp):
    # the same trace and pool: a per-request cap (compression) keeps more requests running than
    # letting every request grow its full cache (a cap far above any length)
    rng = np.random.default_rng(5)
    n = 48
    prompts = rng.integers(16, 128, size=n)
    gens = rng.integers(800, 1600, size=n)
    # capped: every request holds a slot, so every one can compress; uncapped: one protected
    # request and recompute-preemption of the rest when memory runs out
    capped, hist_c, steps_c = _run(zp, prompts, gens, pool=1200, n_max=12, b=16, M=n, check=False)
    full, hist_f, steps_f = _run(zp, prompts, gens, pool=1200, n_max=10_000, b=16, M=1, check=False)
    assert capped["finished"] == full["finished"] == n
    assert np.mean(hist_c) > 1.5 * np.mean(hist_f)
    assert steps_c < steps_f
