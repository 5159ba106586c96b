"""Benchmark of the Compressed-PagedAttention compression pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one compression pass (window attention, Lightning redundancy, combined score,
per-head top-k, global-score update, in-place compaction / target-block writes) over every
(request, layer, kv head) unit of the batch, in one fused launch, followed by the deferred
release of the last blocks.  Default workload: the Llama-3-8B-shaped batch (64 requests x 32
layers, 32/8 heads, d 128, b 16, N_max 128, w 32) = 2048 compressions per step.

Compaction is destructive, so before every step the pool and the global scores are restored
from a pristine device copy, outside the timed CUDA events; the 17 GB restore also evicts L2.
Rank 0 prints one JSON line.  With torchrun (N > 1) every rank compresses its own batch of
the same shape (data-parallel by request, no exchange step) and the time is the max over
ranks.  `--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressions/s (request·layer) and achieved HBM GB/s vs GB300 roofline"


# ------------------------------------------------------------------ helpers ----------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------------ algorithmic bytes -------

def algorithmic_bytes(batch, keep):
    """Bytes the pass must move, per step (one launch).

    K read once: L*d*2 per head; Q read once: w*G_q*d*2 per head; global score read L*4 and
    written L*4 per head; for every moved survivor (destination physical slot differs from the
    source slot): V read + K write + V write = 3*d*2 (moved K comes from shared memory, no
    second read); block tables: 2*n_max*4 per (request, layer).
    """
    import torch
    wl = batch.wl
    R, nl, Hkv, d, b, w = (batch.inp.num_compress, wl.num_layers, wl.num_kv_heads, wl.head_dim,
                           wl.block_size, wl.window)
    Gq = wl.num_q_heads // Hkv
    dev = keep.device
    moved_total = 0
    total = 0
    for r in range(R):
        L = int(batch.seq_len[r])
        t = torch.arange(L, device=dev)
        kp = keep[r, :, :, :L].to(torch.int64)                 # [nl, Hkv, L]
        j = torch.cumsum(kp, -1) - 1                           # destination slot of kept t
        src_tab = torch.from_numpy(batch.tables[r]).to(dev).long()
        dst_tab = torch.from_numpy(batch.dst_tables[r]).to(dev).long()
        jj = j.clamp(min=0)
        same = (src_tab[t // b][None, None, :] == dst_tab[jj // b]) & ((t % b)[None, None, :] == jj % b)
        moved_total += int(((kp == 1) & ~same).sum().item())
        total += nl * Hkv * (L * d * 2 + w * Gq * d * 2 + 2 * L * 4) + nl * 2 * ((L + b - 1) // b) * 4
    total += moved_total * 3 * d * 2
    return total, moved_total


# ------------------------------------------------------------------ CPU oracle baseline -----

def _oracle_task(task):
    from oracle import zipage_oracle as O
    pool, tables, seq, qslot, obs_q, gs, params = task
    O.compress_pass(pool, tables, tables, seq, qslot, obs_q, gs, params)
    return 1


def oracle_sample_tasks(inp, batch_pool, requests, layers):
    """Per-compression oracle inputs (one request, one layer, all kv heads), bf16 bit patterns."""
    import numpy as np
    import torch
    from paged_kv_cache_obs_gb300 import synth
    wl = inp.wl
    tasks = []
    for r in requests:
        blocks = torch.from_numpy(inp.block_tables[r, :wl.n_max].astype(np.int64)).to(batch_pool.device)
        for l in layers:
            pool = synth.bf16_bits(batch_pool[l:l + 1, blocks])
            tables = np.arange(wl.n_max, dtype=np.int32)[None]
            s = int(inp.qslot[r])
            obs_q = synth.bf16_bits(inp.obs_q[s:s + 1, l:l + 1])
            gs = inp.global_scores[s:s + 1, l:l + 1].cpu().numpy()
            p = dict(wl.params(), num_layers=1)
            tasks.append((pool, tables, np.array([wl.L], np.int32), np.array([0], np.int32), obs_q, gs, p))
    return tasks


def time_oracle(tasks, cores):
    """Wall time of the oracle over the tasks on `cores` spawned processes (1 BLAS thread each)."""
    import multiprocessing as mp
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_task, tasks[:cores])  # warm the workers (imports), untimed
        t0 = time.perf_counter()
        pool.map(_oracle_task, tasks, chunksize=1)
        return time.perf_counter() - t0


# ------------------------------------------------------------------ our arm -----------------

def run_ours(args):
    import numpy as np
    import torch
    from paged_kv_cache_obs_gb300 import runner, synth, zipage

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    wl = workload_of(args)
    inp = synth.make_inputs(wl, "cuda", seed=synth.seed_of(wl) + 1000 * rank)
    pristine_pool = inp.pool.clone()
    pristine_gs = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    stream = torch.cuda.Stream()
    compressions = inp.num_compress * wl.num_layers

    # algorithmic bytes from one untimed run with the per-token keep flags
    batch.enable_debug()
    with torch.cuda.stream(stream):
        batch.launch(stream=stream)
    assert batch.error(stream) == 0
    alg_bytes, moved = algorithmic_bytes(batch, batch.debug["keep"])
    batch.debug = None

    def restore():
        batch.pool.copy_(pristine_pool)
        batch.gs.copy_(pristine_gs)

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            restore()
            batch.launch(stream=stream)
    stream.synchronize()
    assert batch.error(stream) == 0

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("timed_steps")  # lets a profiler select the timed launches
        for i in range(args.steps):
            with torch.cuda.stream(stream):
                restore()
                starts[i].record(stream)
                batch.launch(stream=stream)
                ends[i].record(stream)
            batch.commit(stream=stream)           # deferred release of the last blocks (host)
            zipage.zp_alloc_drain(batch.alloc)    # ... and undo it for the next identical step
            batch.close()
            batch.alloc = None
            _reset_alloc(batch, inp)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    barrier(world)
    assert batch.error(stream) == 0
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(times) / len(times)
    ms_max = max_over_ranks(ms, world)
    value = compressions * world / (ms_max / 1e3)

    peak, peak_kind = hbm_peak()
    achieved = alg_bytes / (ms / 1e3) / 1e9
    traffic = _ncu_traffic(args.workload, compressions * wl.num_kv_heads)
    # sequences beyond one cluster (longer than 4096 tokens) take the multi-pass form: four
    # launches per pass (its K is read twice; the algorithmic bytes count it once)
    multipass = (batch.max_seq_len or wl.L) > 4096
    # kernels per pass: 1, or the length grouping and one launch per cluster size when the
    # requests' lengths differ, or the four of the multi-pass form
    launches = zipage.zp_compress_kernel_launches(batch.params, batch.max_seq_len, batch.d_nmax is not None)
    if multipass:
        traffic = None
    out = {
        "metric": METRIC, "value": value, "unit": "compressions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 K/V/Q, fp32 scores", "data": "synthetic (seeded)",
        "config": {"workload": workload_name(wl, inp.num_compress),
                   "compressions_per_step": compressions, "units_per_step": compressions * wl.num_kv_heads,
                   "moved_rows_per_step": moved,
                   "l2": "pool + global scores restored from a pristine device copy before every step "
                         "(17 GB, outside the timed events), so L2 is flushed between steps",
                   "parallelism": f"dp{world} (independent batches, no exchange)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": f"{peak_kind} (hbm_gbs burst copy)",
                     "kernel": ("long_stats/long_score/long_select/long_compact (one pass)" if multipass
                                else "compress_kernel" if launches == 1
                                else f"group_by_length_kernel + compress_kernel at {launches - 1} cluster sizes"
                                     " (one pass)"),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "launch_ms_mean": ms, "launch_ms_min": min(times)},
        "gpu_launches": args.steps * launches,
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, wl, inp, pristine_pool, pristine_gs, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = run_cpu_baseline(inp, pristine_pool, pristine_gs)
    batch.close()
    if world == 1 and args.workload == "llama3_8b" and not args.no_secondary:
        # the other single-pass configurations of the list (Qwen2-7B shape, shared prefix) and the
        # first compression after a prefill (requests grouped by length), timed the same way after
        # the headline measurement and reported beside it
        del batch, inp, pristine_pool, pristine_gs
        torch.cuda.empty_cache()
        out["secondary"] = measure_secondary(["qwen2_7b", "shared_prefix", "prefill"], steps=5, warmup=3)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_secondary(names, steps, warmup):
    """The other workloads of the configuration list, timed exactly as the headline one (pool and
    global scores restored from a pristine device copy outside the timed events, CUDA events on
    the launching stream, algorithmic bytes from the kernel's keep flags), a few steps each, so
    that one run of this script reports them beside the headline number."""
    import torch
    from paged_kv_cache_obs_gb300 import runner, synth, zipage
    out = []
    peak, peak_kind = hbm_peak()
    for name in names:
        wl = synth.WORKLOADS[name]
        inp = synth.make_inputs(wl, "cuda")
        pristine_pool, pristine_gs = inp.pool.clone(), inp.global_scores.clone()
        batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
        stream = torch.cuda.Stream()
        batch.enable_debug()
        with torch.cuda.stream(stream):
            batch.launch(stream=stream)
        assert batch.error(stream) == 0
        alg_bytes, moved = algorithmic_bytes(batch, batch.debug["keep"])
        batch.debug = None
        times = []
        with ClockSampler(torch.cuda.current_device()) as clk:
            for i in range(warmup + steps):
                with torch.cuda.stream(stream):
                    batch.pool.copy_(pristine_pool)
                    batch.gs.copy_(pristine_gs)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    batch.launch(stream=stream)
                    e1.record(stream)
                stream.synchronize()
                if i >= warmup:
                    times.append(e0.elapsed_time(e1))
        assert batch.error(stream) == 0
        ms = sum(times) / len(times)
        comps = inp.num_compress * wl.num_layers
        achieved = alg_bytes / (ms / 1e3) / 1e9
        launches = zipage.zp_compress_kernel_launches(batch.params, batch.max_seq_len, batch.d_nmax is not None)
        out.append({"workload": workload_name(wl, inp.num_compress), "steps": steps, "warmup": warmup,
                    "ms_per_step": ms, "value": comps / (ms / 1e3), "unit": "compressions/s",
                    "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                 "frac": achieved / peak, "peak_kind": f"{peak_kind} (hbm_gbs burst copy)",
                                 "algorithmic_bytes_per_launch": alg_bytes, "moved_rows": moved},
                    "gpu_launches": steps * launches, "clocks": clk.summary()})
        batch.close()
        del batch, inp, pristine_pool, pristine_gs
        torch.cuda.empty_cache()
    return out


def _reset_alloc(batch, inp):
    import numpy as np
    from paged_kv_cache_obs_gb300 import zipage
    batch.alloc = zipage.zp_alloc_create(inp.pool.shape[1])
    used = np.nonzero(inp.refcount)[0].astype(np.int32)
    zipage.zp_alloc_reserve(batch.alloc, used)
    extra = np.repeat(np.arange(inp.pool.shape[1], dtype=np.int32), np.maximum(inp.refcount - 1, 0))
    if len(extra):
        zipage.zp_incref(batch.alloc, extra)
    batch.dst_tables = zipage.zp_plan_compress(batch.alloc, batch.tables, inp.wl.n_max)


COMPRESS_SOURCES = ("zp_compress.cu", "zp_compress_common.cuh", "zp_ptx.cuh")


def _code_lines(text):
    """The lines of a C++/CUDA source without // comments, trailing blanks and empty lines."""
    out = []
    for line in text.splitlines():
        quoted, cut = False, len(line)
        for i, ch in enumerate(line):
            if ch == '"' and (i == 0 or line[i - 1] != "\\"):
                quoted = not quoted
            elif not quoted and line.startswith("//", i):
                cut = i
                break
        code = line[:cut].rstrip()
        if code:
            out.append(code)
    return out


def compress_source_sha256():
    """sha256 over the code (comments and blank lines dropped) of the sources compress_kernel is
    compiled from, in a fixed order: a comment edit keeps a traffic record valid, a code edit
    does not."""
    import hashlib
    h = hashlib.sha256()
    for name in COMPRESS_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_obs_gb300", "csrc", name), encoding="utf-8") as f:
            h.update("\n".join(_code_lines(f.read())).encode())
            h.update(b"\0")
    return h.hexdigest()


def _ncu_traffic(workload, units):
    """DRAM bytes per launch of compress_kernel from the committed ncu summary, if it exists,
    was taken on the current kernel source and covers a launch of this many units (the
    workload at its full size); else null."""
    path = os.path.join(ROOT, "profiles", f"compress_kernel_{workload}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256") != compress_source_sha256() or rec.get("units_full_launch") != units:
            return None
        return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        return None


def run_e2e(args, wl, inp, pristine_pool, pristine_gs, world):
    """Same metric through the public API with HOST buffers.  Every step copies the window
    queries, global scores and tables from pinned host memory, plans on the host, and then
    streams the pool through the GPU a few layers at a time: the host-to-device copy of one
    chunk of layers, the compression of the previous chunk (zp_compress over that layer range)
    and the device-to-host copy of the chunk before it run on three streams at once (the link
    is full duplex).  The compacted pool and global scores end in pinned host memory."""
    import numpy as np
    import torch
    from paged_kv_cache_obs_gb300 import runner, zipage
    # the host-resident pool: each step copies it in, compresses, and copies the compacted pool
    # back into the same buffer (one pinned copy per rank keeps the footprint at one pool)
    h_pool = torch.empty(pristine_pool.shape, dtype=pristine_pool.dtype, pin_memory=True)
    h_pool.copy_(pristine_pool)
    h_out = h_pool
    h_q = inp.obs_q.cpu().pin_memory()
    h_gs = pristine_gs.cpu().pin_memory()
    h_gs_out = torch.empty_like(h_gs, pin_memory=True)
    h_tables = torch.from_numpy(inp.block_tables[:inp.num_compress].copy()).pin_memory()
    batch = runner.CompressionBatch(inp, "cuda", pool=torch.empty_like(pristine_pool))
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nl = wl.num_layers
    per = max(1, nl // 16)  # layers per chunk
    chunks = [(c, min(per, nl - c)) for c in range(0, nl, per)]
    ws = [zipage.new_workspace(zipage.zp_compress_workspace_size(batch.params, inp.num_compress, batch.max_seq_len))
          for _ in chunks]  # one error word per call
    steps = max(2, min(args.steps, 5))
    bytes_in = (h_pool.numel() * 2 + h_q.numel() * 2 + h_gs.numel() * 4 + 2 * h_tables.numel() * 4
                + 2 * inp.num_compress * 4)
    bytes_out = h_pool.numel() * 2 + h_gs.numel() * 4

    def step():
        with torch.cuda.stream(s_in):
            batch.obs_q.copy_(h_q, non_blocking=True)
            batch.gs.copy_(h_gs, non_blocking=True)
            batch.d_tables.copy_(h_tables, non_blocking=True)
        _reset_alloc(batch, inp)
        with torch.cuda.stream(s_in):
            batch.d_dst.copy_(torch.from_numpy(batch.dst_tables).pin_memory(), non_blocking=True)
        done = []
        for i, (l0, n) in enumerate(chunks):
            with torch.cuda.stream(s_in):
                batch.pool[l0:l0 + n].copy_(h_pool[l0:l0 + n], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            batch.workspace = ws[i]
            with torch.cuda.stream(s_comp):
                batch.launch(stream=s_comp, layers=(l0, n))
                ev_c = torch.cuda.Event()
                ev_c.record(s_comp)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                h_out[l0:l0 + n].copy_(batch.pool[l0:l0 + n], non_blocking=True)
            done.append(ev_c)
        with torch.cuda.stream(s_comp):
            batch.commit(stream=s_comp)
        s_out.wait_stream(s_comp)
        with torch.cuda.stream(s_out):
            h_gs_out.copy_(batch.gs, non_blocking=True)
        s_out.synchronize()
        s_comp.synchronize()
        zipage.zp_alloc_drain(batch.alloc)
        zipage.zp_alloc_destroy(batch.alloc)
        batch.alloc = None

    step()
    for w_ in ws:
        assert zipage.zp_read_error(w_) == 0
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) / steps, world)
    comp = inp.num_compress * wl.num_layers * world
    return {"value": comp / dt, "unit": "compressions/s", "h2d_bytes_per_step": int(bytes_in),
            "d2h_bytes_per_step": int(bytes_out), "steps": steps, "ms_per_step": dt * 1e3,
            "pipeline": f"{len(chunks)} chunks of {per} layers: copy in, compress, copy out on three streams"}


def run_cpu_baseline(inp, pool, gs):
    wl = inp.wl
    inp.global_scores = gs
    cores = os.cpu_count() or 1
    reqs = list(range(min(4, inp.num_compress)))
    layers = list(range(wl.num_layers))
    tasks = oracle_sample_tasks(inp, pool, reqs, layers)
    t = time_oracle(tasks, cores)
    return {"value": len(tasks) / t, "unit": "compressions/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(tasks)} compressions ({len(reqs)} requests x {len(layers)} layers, all "
                      f"{wl.num_kv_heads} kv heads) of the same workload, fp64 numpy oracle, "
                      f"{cores} spawned processes x 1 BLAS thread",
            "seconds": t}


# ------------------------------------------------------------------ reference arm -----------

def run_mixed(args):
    """Mixed serving step: the slot holders compress on a side stream while decode attention
    (one new token, every layer) runs for the other requests on the main stream.  Reports the
    compression alone, the decode alone, both concurrently, and the overlap they achieve."""
    import numpy as np
    import torch
    from paged_kv_cache_obs_gb300 import runner, synth, zipage
    torch.cuda.set_device(0)
    wl = workload_of(args)
    # the pool of the mixed configuration: 120k blocks of 2 MiB (all layers), as many as fit
    # beside the rest of the step with a margin
    per_block = wl.num_layers * 2 * wl.num_kv_heads * wl.block_size * wl.head_dim * 2
    free, _ = torch.cuda.mem_get_info()
    nb = min(args.pool_blocks, int((free - (24 << 30)) // per_block))
    if nb > 0:
        wl = wl.scaled(pool_blocks=nb)
    inp = synth.make_inputs(wl, "cuda")
    R = inp.num_compress
    # only the compressing requests' blocks change: they alone are restored between steps
    comp_ids = torch.as_tensor(np.unique(inp.block_tables[:R][inp.block_tables[:R] >= 0]), dtype=torch.int64,
                               device="cuda")
    pristine = inp.pool.index_select(1, comp_ids)
    gs0 = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    p = wl.params()
    nd = wl.num_decode
    dec_tables = torch.from_numpy(np.ascontiguousarray(inp.block_tables[R:])).cuda()
    dec_seq = torch.from_numpy(np.ascontiguousarray(inp.seq_len[R:])).cuda()
    outs = torch.empty((wl.num_layers, nd, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = zipage.new_workspace(zipage.zp_paged_decode_workspace_size(p, nd, wl.n_max))
    # decode (the user-facing tokens) on a high-priority stream, compression on a normal one:
    # as SMs free up, the block scheduler serves decode first (9.45 ms against 9.52 ms a step
    # with equal priorities)
    side, main = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1)  # lower = higher

    def compress():
        batch.launch(stream=side)

    def decode():
        for l in range(wl.num_layers):
            zipage.zp_paged_decode_attn(batch.pool, l, inp.decode_q[l], dec_tables, dec_seq, outs[l], p, ws,
                                        stream=main)

    def timed(fn_c, fn_d):
        batch.pool.index_copy_(1, comp_ids, pristine)
        batch.gs.copy_(gs0)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        ec, ed = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        side.wait_event(e0)
        if fn_c:
            fn_c()
        ec.record(side)
        if fn_d:
            fn_d()
        ed.record(main)
        torch.cuda.synchronize()
        return max(e0.elapsed_time(ec), e0.elapsed_time(ed))

    for _ in range(args.warmup):
        timed(compress, decode)
    tc = np.median([timed(compress, None) for _ in range(args.steps)])
    td = np.median([timed(None, decode) for _ in range(args.steps)])
    torch.cuda.nvtx.range_push("timed_steps")  # the combined steps, for a profiler's launch list
    tb = np.median([timed(compress, decode) for _ in range(args.steps)])
    torch.cuda.nvtx.range_pop()
    assert batch.error(side) == 0 and zipage.zp_read_error(ws, main) == 0
    dec_tokens = int(inp.seq_len[R:].sum())
    dec_bytes = dec_tokens * wl.num_kv_heads * wl.head_dim * 2 * 2 * wl.num_layers
    out = {"metric": METRIC, "value": R * wl.num_layers / (tb / 1e3), "unit": "compressions/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": tb,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded)",
           "config": {"workload": f"mixed: {R} compressing + {nd} decoding requests, {wl.num_layers} layers, "
                                  f"pool {inp.pool.shape[1]} blocks",
                      "note": "one step = compression pass on a side stream + decode of every layer on the main stream"},
           "mixed": {"compress_ms": tc, "decode_ms": td, "both_ms": tb,
                     "overlap_frac": (tc + td - tb) / min(tc, td),
                     "decode_hbm_gbs": dec_bytes / (td / 1e3) / 1e9, "decode_tokens_per_layer": dec_tokens},
           "gpu_launches": 1 + wl.num_layers * zipage.zp_paged_decode_kernel_launches(p, nd, dec_tables.shape[1])}
    print(json.dumps(out), flush=True)
    batch.close()


def workload_name(wl, num_compress):
    """The workload as both arms name it in `config`."""
    return (f"{wl.name}: {num_compress} requests x {wl.num_layers} layers, Hq {wl.num_q_heads}/Hkv "
            f"{wl.num_kv_heads}, d {wl.head_dim}, b {wl.block_size}, N_max {wl.n_max}, w {wl.window}")


def workload_of(args):
    from paged_kv_cache_obs_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.requests:
        wl = wl.scaled(num_requests=args.requests)
    if args.layers:
        wl = wl.scaled(num_layers=args.layers)
    return wl


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from paged_kv_cache_obs_gb300 import synth
    wl = workload_of(args)
    # the same inputs as our arm, drawn on the CPU for the sampled requests only
    small = wl.scaled(num_requests=2)
    inp = synth.make_inputs(small, "cpu", seed=synth.seed_of(wl))
    cores = os.cpu_count() or 1
    per_step = max(cores, 16)
    tasks = oracle_sample_tasks(inp, inp.pool, [0, 1], list(range(wl.num_layers)))
    tasks = (tasks * ((per_step + len(tasks) - 1) // len(tasks)))[:per_step]
    for _ in range(args.warmup):
        time_oracle(tasks[:cores], cores)
    times = [time_oracle(tasks, cores) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = len(tasks) / t
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "compressions/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": workload_name(wl, wl.num_requests),
                      "compressions_per_step": wl.num_requests * wl.num_layers,
                      "units_per_step": wl.num_requests * wl.num_layers * wl.num_kv_heads,
                      "parallelism": "host cores (the fp64 oracle; rank 0 only)"},
           "cpu_baseline": {"value": value, "unit": "compressions/s", "cores": cores, "kind": "oracle",
                            "sample": f"{per_step} compressions per step (request x layer, all kv heads) of "
                                      f"requests 0 and 1, timed and scaled to compressions/s"},
           "e2e": {"value": value, "unit": "compressions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ablation(args):
    """The Lightning ablation: the original all-pairs redundancy kernel alone against the whole
    fused compression pass (whose redundancy is the Lightning form) on the same units, one GPU.
    Defaults to 4 requests of the workload (the all-pairs kernel is O(L^2 d) per head)."""
    import numpy as np
    import torch
    from paged_kv_cache_obs_gb300 import runner, synth, zipage

    torch.cuda.set_device(0)
    if not args.requests:
        args.requests = 4
    wl = workload_of(args)
    inp = synth.make_inputs(wl, "cuda")
    pristine_pool = inp.pool.clone()
    pristine_gs = inp.global_scores.clone()
    batch = runner.CompressionBatch(inp, "cuda", pool=inp.pool)
    stream = torch.cuda.Stream()
    p = wl.params()
    R = inp.num_compress
    L = batch.max_seq_len or wl.L
    redund = torch.empty((R, wl.num_layers, wl.num_kv_heads, L), device="cuda")
    ws = zipage.new_workspace(zipage.zp_redundancy_workspace_size(p, R, batch.max_seq_len))

    def timed(fn):
        ts = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                batch.pool.copy_(pristine_pool)
                batch.gs.copy_(pristine_gs)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
        return float(np.mean(ts))

    ms_pass = timed(lambda: batch.launch(stream=stream))
    assert batch.error(stream) == 0
    ms_ap = timed(lambda: zipage.zp_redundancy_all_pairs(batch.pool, batch.d_tables, batch.d_seq, redund, p, ws,
                                                         stream=stream, max_seq_len=batch.max_seq_len))
    assert zipage.zp_read_error(ws, stream) == 0
    units = R * wl.num_layers * wl.num_kv_heads
    seq = np.asarray(inp.seq_len[:R], np.float64)
    flops = float((2.0 * seq * seq * wl.head_dim).sum()) * wl.num_layers * wl.num_kv_heads
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak, tkind = float(json.load(f)["bf16_tflops"]), "measured (bf16_tflops burst)"
    except (OSError, KeyError, ValueError):
        tpeak, tkind = 1900.0, "fallback"
    out = {"metric": "all-pairs redundancy vs the fused Lightning pass", "ablation": "lightning_vs_all_pairs",
           "unit": "ms", "steps": args.steps, "warmup": args.warmup, "data": "synthetic (seeded)",
           "config": {"workload": f"{wl.name}: {R} requests x {wl.num_layers} layers, {units} head units, L {L}"},
           "fused_pass_ms": ms_pass, "all_pairs_redundancy_ms": ms_ap, "ratio": ms_ap / ms_pass,
           "all_pairs_roofline": {"bound": "tensor", "achieved": flops / ms_ap / 1e9, "peak": tpeak,
                                  "unit": "TFLOP/s", "frac": flops / ms_ap / 1e9 / tpeak, "peak_kind": tkind,
                                  "flops_per_launch": flops}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other configurations reported beside the headline workload")
    ap.add_argument("--requests", type=int, default=0, help="override the workload's request count (profiling)")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--pool-blocks", type=int, default=120000,
                    help="mixed workload: pool size in blocks (capped by free device memory; 0 = just enough)")
    ap.add_argument("--ablation", choices=["all_pairs"], default=None,
                    help="time the original all-pairs redundancy against the fused Lightning pass")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.ablation:
        run_ablation(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.workload == "mixed":
        run_mixed(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
