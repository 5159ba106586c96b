"""Comparison of a compression result against the oracle.  TEST INFRASTRUCTURE ONLY.

Inputs are plain numpy arrays (bf16 bit patterns as uint16, fp32 scores); nothing here
touches the CUDA path.  The acceptance rule:

* attention, redundancy, combined score and carried global score: |x - x_ref| <= 1e-3*|x_ref|
  + 1e-6 (fp32 results against fp64; the absolute floor covers values near zero, e.g. a
  score under cancellation);
* selection: the kernel's kept set must be exactly what the oracle's selection rule gives on
  the kernel's own fp32 scores (the decision taken in the kernel's precision), and may differ
  from the oracle's fp64 selection only for tokens whose oracle score lies within twice that
  tolerance of the oracle's keep/evict boundary (a kept/evicted pair can swap only if the two
  oracle scores differ by at most the sum of their two tolerances);
* compaction: given the kernel's kept set, every compacted K/V row is bit-identical to the
  input row it came from, and every byte of the pool that is not a destination row is
  unchanged.
"""
from __future__ import annotations

import numpy as np

from . import zipage_oracle as O

RTOL = 1e-3
ATOL = 1e-6


def within_tol(x, ref):
    """Elementwise: |x - ref| <= RTOL*|ref| + ATOL for a finite reference; an infinite
    reference (a protected window token's score, fr 2.A) must be matched exactly."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    with np.errstate(invalid="ignore"):
        close = np.abs(x - ref) <= RTOL * np.abs(ref) + ATOL
    return np.where(np.isfinite(ref), close, x == ref)


def assert_close(name, x, ref, where=""):
    ok = within_tol(x, ref)
    if not ok.all():
        i = int(np.nonzero(~ok)[0][0])
        raise AssertionError(f"{name}{where}: {int((~ok).sum())} of {ok.size} outside tolerance; "
                             f"first at {i}: got {float(np.ravel(x)[i])!r}, want {float(np.ravel(ref)[i])!r}")


def check_selection(keep_gpu, S_gpu, S_ref, k, where=""):
    """keep_gpu: 0/1 per token; S_gpu fp32 kernel scores; S_ref fp64 oracle scores."""
    src_gpu = np.nonzero(np.asarray(keep_gpu))[0]
    assert len(src_gpu) == k, f"kept {len(src_gpu)} != {k}{where}"
    same_precision = O.select_keep(np.asarray(S_gpu, np.float32).astype(np.float64), k)
    assert np.array_equal(src_gpu, same_precision), f"selection differs from the rule on kernel scores{where}"
    src_ref = O.select_keep(S_ref, k)
    diff = np.setxor1d(src_gpu, src_ref)
    if len(diff):
        order = sorted(range(len(S_ref)), key=lambda t: (-S_ref[t], t))
        s_k = S_ref[order[k - 1]]
        s_k1 = S_ref[order[k]] if k < len(S_ref) else s_k
        lo = s_k1 - 2 * (RTOL * abs(s_k1) + ATOL)
        hi = s_k + 2 * (RTOL * abs(s_k) + ATOL)
        for t in diff:
            assert lo <= S_ref[t] <= hi, (f"token {t} selected differently far from the boundary{where}: "
                                          f"S={S_ref[t]!r}, boundary [{s_k1!r}, {s_k!r}]")
    return src_gpu


def expected_pool(pool_in, tables, dst_tables, srcs, b):
    """Pool after compaction for the given kept sets: srcs[(r, layer, h)] = kept positions."""
    out = pool_in.copy()
    for (r, l, h), src in srcs.items():
        for j, t in enumerate(src):
            sb, sr = int(tables[r][t // b]), t % b
            db, dr = int(dst_tables[r][j // b]), j % b
            out[l, db, :, h, dr] = pool_in[l, sb, :, h, sr]
    return out


def check_units(units, pool_in, obs_q, gs_in, tables, dst_tables, seq_len, qslot, params,
                dbg_gpu, gs_out, pool_out=None, full_pool=False, n_max_per_req=None):
    """Checks the given units against the oracle.

    dbg_gpu: dict of numpy arrays attn/redund/score/keep shaped [R, layers, Hkv, L].
    gs_out: kernel's global scores after the pass [M, layers, Hkv, L].
    pool_out: kernel's pool after the pass (uint16); with full_pool=True every byte of it is
    compared with the expected pool (requires units to cover every unit).
    Returns the number of tokens whose selection differs from the fp64 oracle.
    """
    b = params["block_size"]
    _, _, ref = O.compress_pass(pool_in, tables, dst_tables, seq_len, qslot, obs_q, gs_in, params,
                                units=units, n_max_per_req=n_max_per_req)
    srcs = {}
    ndiff = 0
    for (r, l, h) in units:
        u = ref[(r, l, h)]
        where = f" at unit (r={r}, layer={l}, h={h})"
        L = int(seq_len[r])
        k = ((int(n_max_per_req[r]) if n_max_per_req is not None else params["n_max"]) - 1) * b
        assert_close("attn", dbg_gpu["attn"][r, l, h][:L], u["attn"], where)
        assert_close("redundancy", dbg_gpu["redund"][r, l, h][:L], u["R"], where)
        assert_close("score", dbg_gpu["score"][r, l, h][:L], u["S"], where)
        src = check_selection(dbg_gpu["keep"][r, l, h][:L], dbg_gpu["score"][r, l, h][:L], u["S"], k, where)
        ndiff += len(np.setxor1d(src, u["src"]))
        srcs[(r, l, h)] = src
        s = int(qslot[r])
        g_want = O.global_update(gs_in[s, l, h, :L].astype(np.float64), u["attn"], src, params["decay"], L)
        assert_close("global score", gs_out[s, l, h, :k], g_want[:k], where)
        assert (gs_out[s, l, h, k:L] == 0).all(), f"global-score tail not zero{where}"
        if pool_out is not None and not full_pool:
            kin = O.gather_rows(pool_in, l, 0, h, tables[r], L, b)
            vin = O.gather_rows(pool_in, l, 1, h, tables[r], L, b)
            kout = O.gather_rows(pool_out, l, 0, h, dst_tables[r], k, b)
            vout = O.gather_rows(pool_out, l, 1, h, dst_tables[r], k, b)
            assert np.array_equal(kout, kin[src]), f"compacted K not bit-exact{where}"
            assert np.array_equal(vout, vin[src]), f"compacted V not bit-exact{where}"
    if full_pool:
        want = expected_pool(pool_in, tables, dst_tables, srcs, b)
        bad = np.nonzero((want != pool_out).reshape(-1))[0]
        assert len(bad) == 0, f"{len(bad)} pool values differ from the expected compacted pool"
    return ndiff
