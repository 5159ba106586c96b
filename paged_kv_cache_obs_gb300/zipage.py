"""ctypes binding of libzipage.so — argument marshalling only.

Every function here has the name of the C entry point it calls (include/zipage.h) and does
nothing but turn tensors into pointers, fill the C structs and raise on a non-OK status.  All
computation of the compression pass and of decode attention runs in the library's CUDA
kernels; there is no fallback: if the library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libzipage.so")

ZP_OK = 0
ZP_ERR_INVALID_ARG = 1
ZP_ERR_NO_BLOCKS = 2
ZP_ERR_BAD_TABLE = 3
ZP_ERR_TIMEOUT = 4
ZP_ERR_CUDA = 5
ZP_ERR_UNSUPPORTED = 6
ZP_ERR_TOO_LARGE = 7
_NAMES = {0: "ZP_OK", 1: "ZP_ERR_INVALID_ARG", 2: "ZP_ERR_NO_BLOCKS", 3: "ZP_ERR_BAD_TABLE",
          4: "ZP_ERR_TIMEOUT", 5: "ZP_ERR_CUDA", 6: "ZP_ERR_UNSUPPORTED", 7: "ZP_ERR_TOO_LARGE"}


class ZipageError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} returned {_NAMES.get(status, status)}")
        self.status = status


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libzipage.so is not built ({_LIB_PATH}); run __graft_entry__.build() "
                      "or python -m paged_kv_cache_obs_gb300.build")
lib = ctypes.CDLL(_LIB_PATH)


class zp_params(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("n_max", ctypes.c_int32), ("window", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("decay", ctypes.c_float),
                ("scale", ctypes.c_float), ("protect_window", ctypes.c_int32),
                ("causal", ctypes.c_int32)]


class zp_kv_pool(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("num_blocks", ctypes.c_int64)]


class zp_seq_meta(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("seq_len", ctypes.c_void_p), ("qslot", ctypes.c_void_p),
                ("dst_tables", ctypes.c_void_p), ("max_seq_len", ctypes.c_int32),
                ("n_max_per_req", ctypes.c_void_p), ("layer_begin", ctypes.c_int32),
                ("layer_count", ctypes.c_int32)]


class zp_debug(ctypes.Structure):
    _fields_ = [("attn", ctypes.c_void_p), ("redund", ctypes.c_void_p),
                ("score", ctypes.c_void_p), ("keep", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_I32P = ctypes.POINTER(ctypes.c_int32)


def _sig(name, res, args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = args
    return f


_sig("zp_compress", _I32, [ctypes.POINTER(zp_kv_pool), _P, ctypes.POINTER(zp_seq_meta), _P, _I32, _P,
                           ctypes.POINTER(zp_params), ctypes.POINTER(zp_debug), _P, _SZ, _P])
_sig("zp_compress_workspace_size", _SZ, [ctypes.POINTER(zp_params), _I32, _I32])
_sig("zp_test_compress_stalled", _I32, [ctypes.POINTER(zp_kv_pool), _P, ctypes.POINTER(zp_seq_meta), _P, _I32, _P,
                                        ctypes.POINTER(zp_params), _P, _SZ, _I64, _P])
_sig("zp_compress_kernel_launches", _I32, [ctypes.POINTER(zp_params), _I32, _I32])
_sig("zp_paged_decode_attn", _I32, [ctypes.POINTER(zp_kv_pool), _I32, _P, _P, _P, _I32, _I32, _P,
                                    ctypes.POINTER(zp_params), _P, _SZ, _P])
_sig("zp_paged_decode_workspace_size", _SZ, [ctypes.POINTER(zp_params), _I32, _I32])
_sig("zp_paged_decode_kernel_launches", _I32, [ctypes.POINTER(zp_params), _I32, _I32])
_sig("zp_paged_decode_attn_static", _I32, [ctypes.POINTER(zp_kv_pool), _I32, _P, _P, _P, _I32, _I32, _P,
                                           ctypes.POINTER(zp_params), _P, _P])
_sig("zp_test_decode_stalled", _I32, [ctypes.POINTER(zp_kv_pool), _I32, _P, _P, _P, _I32, _I32, _P,
                                      ctypes.POINTER(zp_params), _P, _SZ, _I64, _P])
_sig("zp_redundancy_all_pairs", _I32, [ctypes.POINTER(zp_kv_pool), _P, ctypes.POINTER(zp_seq_meta),
                                       ctypes.POINTER(zp_params), _P, _P, _SZ, _P])
_sig("zp_redundancy_workspace_size", _SZ, [ctypes.POINTER(zp_params), _I32, _I32])
_sig("zp_read_error", _I32, [_P, _P, _I32P])
_sig("zp_alloc_create", _I32, [_I64, ctypes.POINTER(_P)])
_sig("zp_alloc_destroy", None, [_P])
_sig("zp_alloc_blocks", _I32, [_P, _I32, _P])
_sig("zp_alloc_reserve", _I32, [_P, _P, _I32])
_sig("zp_incref", _I32, [_P, _P, _I32])
_sig("zp_decref", _I32, [_P, _P, _I32])
_sig("zp_decref_after", _I32, [_P, _P, _I32, _P])
_sig("zp_alloc_poll", _I32, [_P])
_sig("zp_alloc_drain", _I32, [_P])
_sig("zp_alloc_inject_failure", _I32, [_P, _I64])
_sig("zp_refcount", _I32, [_P, _I32])
_sig("zp_num_free", _I64, [_P])
_sig("zp_num_pending", _I64, [_P])
_sig("zp_plan_compress", _I32, [_P, _P, _I32, _I32, _I32, _P])
_sig("zp_commit_compress", _I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P])
_sig("zp_plan_compress_budgets", _I32, [_P, _P, _I32, _I32, _P, _P])
_sig("zp_commit_compress_budgets", _I32, [_P, _P, _P, _I32, _I32, _P, _I32, _I32, _P, _P])
_sig("zp_version", _I32, [])


class zp_sched_config(ctypes.Structure):
    _fields_ = [("n_max", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("max_running", ctypes.c_int32)]


class zp_sched_plan(ctypes.Structure):
    _fields_ = [("num_decode", ctypes.c_int32), ("decode_ids", _I32P), ("num_compress", ctypes.c_int32),
                ("compress_ids", _I32P), ("num_prefill", ctypes.c_int32), ("prefill_ids", _I32P),
                ("num_preempted", ctypes.c_int32), ("preempted_ids", _I32P), ("restricted", ctypes.c_int32)]


class zp_sched_request_info(ctypes.Structure):
    _fields_ = [("state", ctypes.c_int32), ("seq_len", ctypes.c_int32), ("generated", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("table", _I32P), ("has_slot", ctypes.c_int32),
                ("preemptions", ctypes.c_int32)]


class zp_sched_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "submitted", "admitted", "finished", "decoded_tokens",
                                               "compressions", "preemptions", "slot_waits", "restricted_steps",
                                               "blocks_in_use")] + [("running", ctypes.c_int32)]


_sig("zp_sched_create", _I32, [_P, ctypes.POINTER(zp_sched_config), ctypes.POINTER(_P)])
_sig("zp_sched_destroy", None, [_P])
_sig("zp_sched_submit", _I32, [_P, _I32, _I32, _I32P])
_sig("zp_sched_step", _I32, [_P, ctypes.POINTER(zp_sched_plan)])
_sig("zp_sched_request", _I32, [_P, _I32, ctypes.POINTER(zp_sched_request_info)])
_sig("zp_sched_get_stats", _I32, [_P, ctypes.POINTER(zp_sched_stats)])


def _check(fn, status):
    if status != ZP_OK:
        raise ZipageError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_params(p: dict) -> zp_params:
    return zp_params(p["num_layers"], p["num_q_heads"], p["num_kv_heads"], p["head_dim"],
                     p["block_size"], p["n_max"], p["window"], p["alpha"], p["beta"], p["decay"],
                     p["scale"], int(p["protect_window"]), int(p["causal"]))


def _i32_array(a):
    """Contiguous host int32 buffer (numpy array or sequence) -> (ctypes array, keepalive)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr.ctypes.data_as(ctypes.c_void_p), arr


# ------------------------------------------------------------------ compression pass --------

def zp_compress_workspace_size(params: dict, num_requests: int, max_seq_len: int = 0) -> int:
    return lib.zp_compress_workspace_size(ctypes.byref(make_params(params)), num_requests, max_seq_len)


def zp_compress_kernel_launches(params: dict, max_seq_len: int = 0, per_request_budgets: bool = False) -> int:
    return lib.zp_compress_kernel_launches(ctypes.byref(make_params(params)), max_seq_len, int(per_request_budgets))


def zp_compress(pool, block_tables, seq_len, qslot, dst_tables, obs_q, global_scores, params: dict,
                workspace, debug: dict | None = None, stream=None, max_seq_len: int = 0, n_max_per_req=None,
                layers: tuple | None = None):
    """Queues the compression pass; tensors are device tensors (see include/zipage.h).
    max_seq_len: the longest seq_len of the call (0: every request holds n_max*b tokens).
    n_max_per_req: optional device int32 [R] of per-request block budgets.
    layers: optional (layer_begin, layer_count) to compress only those layers."""
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    lb, lc = layers if layers is not None else (0, 0)
    meta = zp_seq_meta(block_tables.shape[0], block_tables.shape[1], seq_len.data_ptr(),
                       qslot.data_ptr(), dst_tables.data_ptr(), max_seq_len,
                       None if n_max_per_req is None else n_max_per_req.data_ptr(), lb, lc)
    dbg = None
    if debug:
        dbg = zp_debug(*(debug[k].data_ptr() if debug.get(k) is not None else None
                         for k in ("attn", "redund", "score", "keep")))
    st = lib.zp_compress(ctypes.byref(kv), _ptr(block_tables), ctypes.byref(meta), _ptr(obs_q),
                         obs_q.shape[0], _ptr(global_scores), ctypes.byref(make_params(params)),
                         ctypes.byref(dbg) if dbg is not None else None, _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check("zp_compress", st)


def zp_test_compress_stalled(pool, block_tables, seq_len, qslot, dst_tables, obs_q, global_scores, params: dict,
                             workspace, stall_limit_ns: int, max_seq_len: int, stream=None, n_max_per_req=None):
    """Test hook of the bounded waits: the multi-pass compression (max_seq_len > 4096) whose
    statistics CTAs first wait, at most stall_limit_ns, on a barrier nothing completes, and so
    report ZP_ERR_TIMEOUT."""
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    meta = zp_seq_meta(block_tables.shape[0], block_tables.shape[1], seq_len.data_ptr(),
                       qslot.data_ptr(), dst_tables.data_ptr(), max_seq_len,
                       None if n_max_per_req is None else n_max_per_req.data_ptr(), 0, 0)
    st = lib.zp_test_compress_stalled(ctypes.byref(kv), _ptr(block_tables), ctypes.byref(meta), _ptr(obs_q),
                                      obs_q.shape[0], _ptr(global_scores), ctypes.byref(make_params(params)),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      int(stall_limit_ns), _stream(stream))
    _check("zp_test_compress_stalled", st)


# ------------------------------------------------------------------ all-pairs redundancy -----

def zp_redundancy_workspace_size(params: dict, num_requests: int, max_seq_len: int = 0) -> int:
    return lib.zp_redundancy_workspace_size(ctypes.byref(make_params(params)), num_requests, max_seq_len)


def zp_redundancy_all_pairs(pool, block_tables, seq_len, redund, params: dict, workspace, stream=None,
                            max_seq_len: int = 0):
    """Queues the original all-pairs redundancy (the Lightning ablation) into redund
    [R][layers][H_kv][L_max] fp32 (see include/zipage.h)."""
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    meta = zp_seq_meta(block_tables.shape[0], block_tables.shape[1], seq_len.data_ptr(), None, None,
                       max_seq_len, None)
    st = lib.zp_redundancy_all_pairs(ctypes.byref(kv), _ptr(block_tables), ctypes.byref(meta),
                                     ctypes.byref(make_params(params)), _ptr(redund), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check("zp_redundancy_all_pairs", st)


# ------------------------------------------------------------------ decode attention ---------

def zp_paged_decode_workspace_size(params: dict, B: int, max_blocks: int) -> int:
    return lib.zp_paged_decode_workspace_size(ctypes.byref(make_params(params)), B, max_blocks)


def zp_paged_decode_kernel_launches(params: dict, B: int, max_blocks: int) -> int:
    return lib.zp_paged_decode_kernel_launches(ctypes.byref(make_params(params)), B, max_blocks)


def zp_paged_decode_attn(pool, layer: int, q, block_tables, seq_lens, out, params: dict, workspace,
                         stream=None):
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    st = lib.zp_paged_decode_attn(ctypes.byref(kv), layer, _ptr(q), _ptr(block_tables), _ptr(seq_lens),
                                  q.shape[0], block_tables.shape[1], _ptr(out),
                                  ctypes.byref(make_params(params)), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check("zp_paged_decode_attn", st)


def zp_test_decode_stalled(pool, layer: int, q, block_tables, seq_lens, out, params: dict, workspace,
                           stall_limit_ns: int, stream=None):
    """Test hook of the bounded waits: decode attention whose kernel first waits, at most
    stall_limit_ns, on a barrier nothing completes, and so reports ZP_ERR_TIMEOUT."""
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    st = lib.zp_test_decode_stalled(ctypes.byref(kv), layer, _ptr(q), _ptr(block_tables), _ptr(seq_lens),
                                    q.shape[0], block_tables.shape[1], _ptr(out),
                                    ctypes.byref(make_params(params)), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), int(stall_limit_ns),
                                    _stream(stream))
    _check("zp_test_decode_stalled", st)


def zp_paged_decode_attn_static(pool, layer: int, q, block_tables, seq_lens, out, params: dict,
                                dev_status=None, stream=None):
    """Decode attention whose scratch is the library's fixed device array: nothing is
    allocated, so callers without a device allocator can use it (see include/zipage.h).
    dev_status: optional device int32 tensor receiving the device-side status."""
    kv = zp_kv_pool(pool.data_ptr(), pool.shape[1])
    st = lib.zp_paged_decode_attn_static(ctypes.byref(kv), layer, _ptr(q), _ptr(block_tables), _ptr(seq_lens),
                                         q.shape[0], block_tables.shape[1], _ptr(out),
                                         ctypes.byref(make_params(params)), _ptr(dev_status), _stream(stream))
    _check("zp_paged_decode_attn_static", st)


def zp_read_error(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("zp_read_error", lib.zp_read_error(_ptr(workspace), _stream(stream), ctypes.byref(out)))
    return out.value


def new_workspace(nbytes: int, device="cuda"):
    """Device workspace of at least nbytes (256-byte aligned: torch allocations are)."""
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ allocator (host) --------

def zp_alloc_create(num_blocks: int):
    h = ctypes.c_void_p()
    _check("zp_alloc_create", lib.zp_alloc_create(num_blocks, ctypes.byref(h)))
    return h


def zp_alloc_destroy(a):
    lib.zp_alloc_destroy(a)


def zp_alloc_blocks(a, n: int):
    import numpy as np
    ids = np.zeros(max(n, 1), dtype=np.int32)
    _check("zp_alloc_blocks", lib.zp_alloc_blocks(a, n, ids.ctypes.data_as(ctypes.c_void_p)))
    return ids[:n]


def zp_alloc_reserve(a, ids):
    p, keep = _i32_array(ids)
    _check("zp_alloc_reserve", lib.zp_alloc_reserve(a, p, len(keep)))


def zp_incref(a, ids):
    p, keep = _i32_array(ids)
    _check("zp_incref", lib.zp_incref(a, p, len(keep)))


def zp_decref(a, ids):
    p, keep = _i32_array(ids)
    _check("zp_decref", lib.zp_decref(a, p, len(keep)))


def zp_decref_after(a, ids, stream=None):
    p, keep = _i32_array(ids)
    st = None if stream is False else _stream(stream)
    _check("zp_decref_after", lib.zp_decref_after(a, p, len(keep), st))


def zp_alloc_poll(a):
    _check("zp_alloc_poll", lib.zp_alloc_poll(a))


def zp_alloc_drain(a):
    _check("zp_alloc_drain", lib.zp_alloc_drain(a))


def zp_alloc_inject_failure(a, nth_call: int):
    _check("zp_alloc_inject_failure", lib.zp_alloc_inject_failure(a, nth_call))


def zp_refcount(a, block_id: int) -> int:
    return lib.zp_refcount(a, block_id)


def zp_num_free(a) -> int:
    return lib.zp_num_free(a)


def zp_num_pending(a) -> int:
    return lib.zp_num_pending(a)


def zp_plan_compress(a, host_tables, n_max: int):
    """host_tables: int32 [R, max_blocks] (numpy) -> destination tables (numpy)."""
    import numpy as np
    t = np.ascontiguousarray(host_tables, dtype=np.int32)
    out = np.zeros_like(t)
    _check("zp_plan_compress", lib.zp_plan_compress(a, t.ctypes.data_as(ctypes.c_void_p), t.shape[0],
                                                    t.shape[1], n_max,
                                                    out.ctypes.data_as(ctypes.c_void_p)))
    return out


def zp_plan_compress_budgets(a, host_tables, n_max_per_req):
    import numpy as np
    t = np.ascontiguousarray(host_tables, dtype=np.int32)
    nm = np.ascontiguousarray(n_max_per_req, dtype=np.int32)
    out = np.zeros_like(t)
    _check("zp_plan_compress_budgets", lib.zp_plan_compress_budgets(
        a, t.ctypes.data_as(ctypes.c_void_p), t.shape[0], t.shape[1], nm.ctypes.data_as(ctypes.c_void_p),
        out.ctypes.data_as(ctypes.c_void_p)))
    return out


def zp_commit_compress_budgets(a, old_tables, new_tables, n_max_per_req, n_max: int, stream=None,
                               block_size: int = 0, seq_len=None):
    import numpy as np
    o = np.ascontiguousarray(old_tables, dtype=np.int32)
    n = np.ascontiguousarray(new_tables, dtype=np.int32)
    nm = np.ascontiguousarray(n_max_per_req, dtype=np.int32)
    sl = None if seq_len is None else np.ascontiguousarray(seq_len, dtype=np.int32)
    st = None if stream is False else _stream(stream)
    _check("zp_commit_compress_budgets", lib.zp_commit_compress_budgets(
        a, o.ctypes.data_as(ctypes.c_void_p), n.ctypes.data_as(ctypes.c_void_p), o.shape[0], o.shape[1],
        nm.ctypes.data_as(ctypes.c_void_p), n_max, block_size,
        None if sl is None else sl.ctypes.data_as(ctypes.c_void_p), st))


def zp_commit_compress(a, old_tables, new_tables, n_max: int, stream=None, block_size: int = 0,
                       seq_len=None):
    """seq_len: host per-request token counts (None: every request holds n_max blocks)."""
    import numpy as np
    o = np.ascontiguousarray(old_tables, dtype=np.int32)
    n = np.ascontiguousarray(new_tables, dtype=np.int32)
    sl = None if seq_len is None else np.ascontiguousarray(seq_len, dtype=np.int32)
    st = None if stream is False else _stream(stream)
    _check("zp_commit_compress", lib.zp_commit_compress(
        a, o.ctypes.data_as(ctypes.c_void_p), n.ctypes.data_as(ctypes.c_void_p), o.shape[0], o.shape[1], n_max,
        block_size, None if sl is None else sl.ctypes.data_as(ctypes.c_void_p), st))


def zp_version() -> int:
    return lib.zp_version()


# ------------------------------------------------------------------ hybrid scheduler (host) --

def zp_sched_create(alloc, n_max: int, block_size: int, num_slots: int, max_running: int = 0):
    h = ctypes.c_void_p()
    cfg = zp_sched_config(n_max, block_size, num_slots, max_running)
    _check("zp_sched_create", lib.zp_sched_create(alloc, ctypes.byref(cfg), ctypes.byref(h)))
    return h


def zp_sched_destroy(s):
    lib.zp_sched_destroy(s)


def zp_sched_submit(s, prompt_len: int, gen_len: int) -> int:
    rid = ctypes.c_int32()
    _check("zp_sched_submit", lib.zp_sched_submit(s, prompt_len, gen_len, ctypes.byref(rid)))
    return rid.value


def zp_sched_step(s) -> dict:
    p = zp_sched_plan()
    _check("zp_sched_step", lib.zp_sched_step(s, ctypes.byref(p)))
    ids = lambda n, ptr: [ptr[i] for i in range(n)]
    return {"decode": ids(p.num_decode, p.decode_ids), "compress": ids(p.num_compress, p.compress_ids),
            "prefill": ids(p.num_prefill, p.prefill_ids), "preempted": ids(p.num_preempted, p.preempted_ids),
            "restricted": bool(p.restricted)}


def zp_sched_request(s, rid: int) -> dict:
    i = zp_sched_request_info()
    _check("zp_sched_request", lib.zp_sched_request(s, rid, ctypes.byref(i)))
    return {"state": i.state, "seq_len": i.seq_len, "generated": i.generated, "num_blocks": i.num_blocks,
            "table": [i.table[k] for k in range(i.num_blocks)], "has_slot": bool(i.has_slot),
            "preemptions": i.preemptions}


def zp_sched_get_stats(s) -> dict:
    st = zp_sched_stats()
    _check("zp_sched_get_stats", lib.zp_sched_get_stats(s, ctypes.byref(st)))
    return {n: getattr(st, n) for n, _ in zp_sched_stats._fields_}
