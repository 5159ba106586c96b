"""C-ABI library: it loads, exports every entry point of include/zipage.h, and its host-side
allocator / planner behave like the literal refcount model (no GPU needed for any of this)."""
import os
import re

import numpy as np
import pytest

from oracle import zipage_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def zp():
    from paged_kv_cache_obs_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_obs_gb300 import zipage
    return zipage


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(zp_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(zp):
    names = _declared_symbols()
    assert len(names) >= 20
    for n in names:
        assert hasattr(zp.lib, n), n
    assert zp.zp_version() == 1


def test_alloc_lowest_first_and_transactional(zp):
    a = zp.zp_alloc_create(8)
    try:
        assert list(zp.zp_alloc_blocks(a, 3)) == [0, 1, 2]
        assert zp.zp_num_free(a) == 5
        with pytest.raises(zp.ZipageError) as e:
            zp.zp_alloc_blocks(a, 6)
        assert e.value.status == zp.ZP_ERR_NO_BLOCKS
        assert zp.zp_num_free(a) == 5            # nothing changed
        zp.zp_decref(a, [1])
        assert zp.zp_refcount(a, 1) == 0
        assert list(zp.zp_alloc_blocks(a, 2)) == [1, 3]
        with pytest.raises(zp.ZipageError):
            zp.zp_decref(a, [5])                  # free block
        with pytest.raises(zp.ZipageError):
            zp.zp_decref(a, [0, 0])               # refcount 1, two decrefs: all-or-nothing
        assert zp.zp_refcount(a, 0) == 1
        assert zp.zp_refcount(a, 99) == -1
    finally:
        zp.zp_alloc_destroy(a)


def test_reserve_incref_and_injected_failure(zp):
    a = zp.zp_alloc_create(10)
    try:
        zp.zp_alloc_reserve(a, [7, 2, 5])
        assert [zp.zp_refcount(a, i) for i in (2, 5, 7)] == [1, 1, 1]
        with pytest.raises(zp.ZipageError):
            zp.zp_alloc_reserve(a, [3, 3])
        with pytest.raises(zp.ZipageError):
            zp.zp_alloc_reserve(a, [2])
        zp.zp_incref(a, [5, 5])
        assert zp.zp_refcount(a, 5) == 3
        zp.zp_alloc_inject_failure(a, 2)
        zp.zp_alloc_blocks(a, 1)                   # first call succeeds
        free_before = zp.zp_num_free(a)
        with pytest.raises(zp.ZipageError) as e:
            zp.zp_alloc_blocks(a, 1)               # second fails, changes nothing
        assert e.value.status == zp.ZP_ERR_NO_BLOCKS and zp.zp_num_free(a) == free_before
        zp.zp_alloc_blocks(a, 1)
    finally:
        zp.zp_alloc_destroy(a)


def _state_from(inp_refcount):
    return {i: int(c) for i, c in enumerate(inp_refcount)}


@pytest.mark.parametrize("prefix", [0, 4])
def test_plan_and_commit_match_refcount_model(zp, prefix):
    rng = np.random.default_rng(prefix)
    NB, R, n_max, mb = 200, 5, 12, 14
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((R, mb), -1, np.int32)
    shared = perm[:prefix]
    nxt = prefix
    for r in range(R):
        tables[r, :prefix] = shared
        tables[r, prefix:n_max] = perm[nxt:nxt + n_max - prefix]
        nxt += n_max - prefix
    model = O.RefcountPool(NB)
    a = zp.zp_alloc_create(NB)
    try:
        used = sorted(set(tables[tables >= 0].tolist()))
        zp.zp_alloc_reserve(a, used)
        for i in used:
            model.refcount[i] = 1
        if prefix:
            extra = list(shared) * R  # R requests + the prefix cache's own reference
            zp.zp_incref(a, extra)
            model.incref(extra)
        dst = zp.zp_plan_compress(a, tables, n_max)
        free = model.free_ids()
        want = tables.copy()
        for r in range(R):
            row, _ = O.plan_dst_table(tables[r], n_max, dict(enumerate(model.refcount)), free)
            want[r, :n_max - 1] = row
        fresh = want[:, :prefix].ravel().tolist()
        for i in fresh:
            model.refcount[i] = 1
        assert np.array_equal(dst, want)
        assert zp.zp_num_free(a) == model.num_free()
        # commit, deferred only by a NULL stream here (host-only): released at once
        zp.zp_commit_compress(a, tables, dst, n_max, stream=False)
        for r in range(R):
            rel = [tables[r, i] for i in range(n_max - 1) if tables[r, i] != dst[r, i]] + [tables[r, n_max - 1]]
            model.decref(rel)
        assert [zp.zp_refcount(a, i) for i in range(NB)] == model.refcount
        # one freed last block per request; shared blocks stay live (prefix-cache reference)
        assert zp.zp_num_free(a) == NB - (R * (n_max - 1) + (prefix and prefix))
        for s in shared:
            assert zp.zp_refcount(a, int(s)) == 1
        # the planner is transactional when blocks run out
        if prefix:
            with pytest.raises(zp.ZipageError):
                zp.zp_incref(a, [999])
            big = dst[:1].copy()
            big[0, n_max - 1] = zp.zp_alloc_blocks(a, 1)[0]   # a new last block
            zp.zp_incref(a, list(big[0, :n_max - 1]))          # make request 0's blocks shared
            zp.zp_alloc_inject_failure(a, 1)
            before = [zp.zp_refcount(a, i) for i in range(NB)]
            with pytest.raises(zp.ZipageError) as e:
                zp.zp_plan_compress(a, big, n_max)
            assert e.value.status == zp.ZP_ERR_NO_BLOCKS
            assert [zp.zp_refcount(a, i) for i in range(NB)] == before
    finally:
        zp.zp_alloc_destroy(a)


def test_invalid_arguments_are_rejected_without_a_gpu(zp):
    p = dict(num_layers=1, num_q_heads=4, num_kv_heads=3, head_dim=64, block_size=16, n_max=8,
             window=8, alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    import ctypes
    kv = zp.zp_kv_pool(None, 0)
    st = zp.lib.zp_compress(ctypes.byref(kv), None, None, None, 1, None,
                            ctypes.byref(zp.make_params(p)), None, None, 0, None)
    assert st == zp.ZP_ERR_INVALID_ARG
    assert zp.zp_compress_workspace_size(p, 4) >= 4
    assert zp.zp_paged_decode_workspace_size(dict(p, num_kv_heads=2), 3, 20) > 256
    # decode launch count: 1 or 2 for valid sizes, 0 otherwise; a request of at most 32 blocks
    # is always one split
    q = dict(p, num_kv_heads=2)
    assert zp.zp_paged_decode_kernel_launches(q, 3, 20) == 1
    assert zp.zp_paged_decode_kernel_launches(q, 3, 4096) in (1, 2)
    assert zp.zp_paged_decode_kernel_launches(q, 0, 20) == 0
    assert zp.zp_paged_decode_kernel_launches(q, 3, 0) == 0


def test_compress_launch_plan_and_workspace_without_a_gpu(zp):
    # The launch-count query follows the cluster sizes a call needs: 256 keys per CTA, so a
    # request of L tokens takes ceil(L / 256) CTAs.  The Llama-3-8B decode trigger (N_max 128,
    # b 16: L = 2048, k = 2032) is one launch; after a prefill to 2048 with N_max 64 (k = 1008)
    # the requests need 4..8 CTAs, so the grouping kernel and 5 launches; with per-request
    # budgets (k_r >= b) any of 1..8; beyond 4096 tokens the four multi-pass kernels.
    p = dict(num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, n_max=128,
             window=32, alpha=0.5, beta=0.5, decay=0.9, scale=0.088, protect_window=1, causal=1)
    assert zp.zp_compress_kernel_launches(p) == 1
    assert zp.zp_compress_kernel_launches(p, 2048) == 1
    assert zp.zp_compress_kernel_launches(dict(p, n_max=64), 2048) == 1 + 5
    assert zp.zp_compress_kernel_launches(dict(p, n_max=64), 1024) == 1   # L = n_max*b: one size
    assert zp.zp_compress_kernel_launches(p, 0, per_request_budgets=True) == 1 + 8
    assert zp.zp_compress_kernel_launches(p, 4096) == 1 + (16 - 8 + 1)
    assert zp.zp_compress_kernel_launches(p, 8192) == 4
    assert zp.zp_compress_kernel_launches(p, 2032) == 0                  # L <= k
    assert zp.zp_compress_kernel_launches(p, 16385) == 0
    assert zp.zp_compress_kernel_launches(dict(p, block_size=8)) == 0
    # workspace: a 512-byte header and the grouped request order (4 bytes per request) up to
    # 4096 tokens, rounded up to 256 bytes
    assert zp.zp_compress_workspace_size(p, 64) == 512 + 256
    assert zp.zp_compress_workspace_size(p, 65) == 512 + 512
    assert zp.zp_compress_workspace_size(p, 0) == 512
    # a call whose workspace is below that size is refused before anything reaches the device
    # (the buffers below are host memory that the call must not touch)
    import ctypes
    import numpy as np
    R = 64
    host = np.zeros(1 << 16, np.uint8)
    ptr = host.ctypes.data
    kv = zp.zp_kv_pool(ptr, 16)
    meta = zp.zp_seq_meta(R, 129, ptr, ptr, ptr, 0, None, 0, 0)
    ws = np.zeros(4096, np.uint8)
    wsp = (ws.ctypes.data + 255) // 256 * 256
    for nbytes, expect in ((256, zp.ZP_ERR_INVALID_ARG), (511 + 256, zp.ZP_ERR_INVALID_ARG)):
        st = zp.lib.zp_compress(ctypes.byref(kv), ctypes.c_void_p(ptr), ctypes.byref(meta), ctypes.c_void_p(ptr),
                                1, ctypes.c_void_p(ptr), ctypes.byref(zp.make_params(p)), None,
                                ctypes.c_void_p(wsp), nbytes, None)
        assert st == expect
    assert not host.any() and not ws.any()


def test_commit_after_prefill_releases_every_block_past_n_max_minus_1(zp):
    a = zp.zp_alloc_create(64)
    try:
        n_max, b = 4, 16
        ids = zp.zp_alloc_blocks(a, 7 + 4)          # request 0: 7 blocks, request 1: 4 blocks
        tables = np.full((2, 8), -1, np.int32)
        tables[0, :7] = ids[:7]
        tables[1, :4] = ids[7:]
        seq = np.array([7 * b - 5, 4 * b], np.int32)  # request 0 left a prefill of 107 tokens
        dst = zp.zp_plan_compress(a, tables, n_max)
        assert np.array_equal(dst, tables)            # nothing shared: in place
        free0 = zp.zp_num_free(a)
        zp.zp_commit_compress(a, tables, dst, n_max, stream=False, block_size=b, seq_len=seq)
        assert zp.zp_num_free(a) == free0 + (7 - 3) + (4 - 3)
        for i in list(ids[3:7]) + [ids[10]]:
            assert zp.zp_refcount(a, int(i)) == 0
        for i in list(ids[:3]) + list(ids[7:10]):
            assert zp.zp_refcount(a, int(i)) == 1
    finally:
        zp.zp_alloc_destroy(a)


def test_plan_and_commit_with_per_request_budgets(zp):
    a = zp.zp_alloc_create(40)
    try:
        # request 0: budget 3 with a shared first block; request 1: budget 5, nothing shared
        ids = zp.zp_alloc_blocks(a, 3 + 5)
        tables = np.full((2, 6), -1, np.int32)
        tables[0, :3] = ids[:3]
        tables[1, :5] = ids[3:8]
        zp.zp_incref(a, [ids[0]])                          # block ids[0] is shared
        dst = zp.zp_plan_compress_budgets(a, tables, [3, 5])
        assert dst[0, 0] != tables[0, 0] and zp.zp_refcount(a, int(dst[0, 0])) == 1   # target block
        assert np.array_equal(dst[0, 1:], tables[0, 1:]) and np.array_equal(dst[1], tables[1])
        free0 = zp.zp_num_free(a)
        zp.zp_commit_compress_budgets(a, tables, dst, [3, 5], 5, stream=False)
        # released: the replaced shared block (decref only), the last block of each request
        assert zp.zp_refcount(a, int(ids[0])) == 1
        assert zp.zp_refcount(a, int(ids[2])) == 0 and zp.zp_refcount(a, int(ids[7])) == 0
        assert zp.zp_num_free(a) == free0 + 2
        with pytest.raises(zp.ZipageError):
            zp.zp_plan_compress_budgets(a, tables, [1, 5])  # a budget below 2
    finally:
        zp.zp_alloc_destroy(a)


def test_host_validation_of_layer_ranges_and_all_pairs(zp):
    """Argument checks that return before any device work (no GPU needed): a layer range past
    the last layer, a negative count, a begin without a count; and the all-pairs redundancy's
    unsupported head sizes and lengths."""
    import ctypes
    p = dict(num_layers=4, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, n_max=8,
             window=8, alpha=0.5, beta=0.5, decay=0.9, scale=0.125, protect_window=1, causal=1)
    fake = 1 << 20  # never dereferenced: the calls fail before touching device memory
    kv = zp.zp_kv_pool(fake, 64)
    params = zp.make_params(p)
    for lb, lc in ((3, 2), (0, -1), (1, 0), (-1, 2)):
        meta = zp.zp_seq_meta(1, 8, fake, fake, fake, 0, None, lb, lc)
        st = zp.lib.zp_compress(ctypes.byref(kv), fake, ctypes.byref(meta), fake, 1, fake, ctypes.byref(params),
                                None, fake, 256, None)
        assert st == zp.ZP_ERR_INVALID_ARG, (lb, lc)
    meta = zp.zp_seq_meta(1, 8, fake, None, None, 0, None, 0, 0)
    bad_d = zp.make_params(dict(p, head_dim=96))
    big = 1 << 30  # a workspace size that passes its check
    assert zp.lib.zp_redundancy_all_pairs(ctypes.byref(kv), fake, ctypes.byref(meta), ctypes.byref(bad_d), fake,
                                          fake, big, None) == zp.ZP_ERR_UNSUPPORTED
    long_meta = zp.zp_seq_meta(1, 400, fake, None, None, 5000, None, 0, 0)
    assert zp.lib.zp_redundancy_all_pairs(ctypes.byref(kv), fake, ctypes.byref(long_meta), ctypes.byref(params),
                                          fake, fake, big, None) == zp.ZP_ERR_UNSUPPORTED
    assert zp.lib.zp_redundancy_all_pairs(ctypes.byref(kv), fake, ctypes.byref(meta), ctypes.byref(params),
                                          fake, fake, 256, None) == zp.ZP_ERR_INVALID_ARG  # workspace too small
    # error word plus one fp32 squared norm per (request, layer, kv head, token)
    assert zp.zp_redundancy_workspace_size(p, 3, 100) == 256 + 3 * 4 * 2 * 100 * 4
