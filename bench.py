"""Benchmark: paged decode attention on one GB300 (or N independent replicas).

One step = one decode step of one attention layer over the batch-64 decode
workload (64 sequences, 16 query / 8 kv heads, head_dim 128, 256-token blocks,
context lengths uniform in [512, 4096], physical blocks shuffled in a 2048-block
pool): the store of the 64 new tokens and the decode, in one launch
(paged_decode_attention_store); the same steps as two launches
(kv_cache_store, then paged_decode_attention) are timed beside it.

Inputs larger than L2: each step reads about 524 MB of K/V (L2 is ~129 MB), and
consecutive steps cycle through three batches whose blocks are disjoint, so no
step finds the previous step's K/V in L2.

Prints one JSON line (rank 0).  `value` is algorithmic HBM bytes per step
(the decode's 4096 B per context token plus q, out, lse and table entries, and
the store's new rows read and written) x steps / device time, in GB/s; the same line
carries KV-tokens/s, the roofline of the step's kernel, the oracle
timed on the host cores (`cpu_baseline`), an end-to-end number through the
public API with host buffers (`e2e`), clocks sampled during the timed region
and extra measurements of the other workloads.

`--impl reference` times the CPU oracle instead, on a bounded sample of the
same workload, and prints the same kind of line with "impl": "reference".
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

_ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, _ROOT)

from paged_kv_cache_214_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak), KV-tokens/s"
WORKLOAD = "decode-b64: B=64, Hq=16, Hkv=8, D=128, block 256, ctx U[512,4096], 2048-block pool"
ROTATIONS = 3
BF16 = 2


def _peaks():
    try:
        with open(os.path.join(_ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic bytes


def decode_bytes(w, unique: bool = False, kv_elem_bytes: int = BF16) -> int:
    """K/V of every context token read once (shared prefix once if `unique`),
    q read, out written, lse written, block-table entries and lengths read.
    `kv_elem_bytes`: 2 for the bf16 cache, 1 for the FP8 one."""
    toks = w.unique_kv_tokens if unique else w.kv_tokens
    kv = toks * w.Hkv * w.D * kv_elem_bytes * 2
    qo = 2 * w.B * w.Hq * w.D * BF16
    lse = w.B * w.Hq * 4
    tables = int(sum(-(-int(L) // w.block_size) for L in w.context_lens)) * 4 + w.B * 4
    return kv + qo + lse + tables


def store_bytes(T: int, Hkv: int, D: int) -> int:
    """T tokens: read k and v rows, write them into the pool, read the slots."""
    return T * Hkv * D * BF16 * 2 * 2 + T * 4


def prefill_flops(w) -> float:
    """4*D per (query row, visible key, head): QK^T and PV multiply-adds."""
    total = 0
    for lq, lk in zip(w.q_lens, w.k_lens):
        # row r sees lk - lq + r + 1 keys
        total += lq * (lk - lq) + lq * (lq + 1) // 2
    return 4.0 * w.D * w.Hq * total


# ----------------------------------------------------------------------------
# clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        self.gpu_id = None
        try:
            props = torch.cuda.get_device_properties(device)
            self.gpu_id = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id,
                                                props.pci_device_id)
        except Exception:
            self.gpu_id = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # nvidia-smi's start-up (library load, device attach) runs before the
        # warm-up, not inside the timed region
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# distributed plumbing (independent replicas; no data-path collective)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# oracle (host) timing


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_sample(w, n_seq: int):
    """Host inputs of the first n_seq sequences (compact pool of their blocks)."""
    seqs = list(range(n_seq))
    tables = w.block_tables[seqs]
    used = tables[tables >= 0].unique()
    remap = torch.full((w.num_blocks,), -1, dtype=torch.int64)
    remap[used.long()] = torch.arange(used.numel())
    idx = used.to(w.k_cache.device).long()
    kc = _bits(w.k_cache.index_select(0, idx)).copy()
    vc = _bits(w.v_cache.index_select(0, idx)).copy()
    t = tables.clone().long()
    t[t >= 0] = remap[t[t >= 0]]
    bs = w.block_size
    slots = []
    for s in w.slot_mapping[seqs].tolist():
        slots.append(int(remap[s // bs]) * bs + s % bs if s >= 0 else -1)
    return dict(q=_bits(w.q[seqs]), k=_bits(w.k_new[seqs]), v=_bits(w.v_new[seqs]),
                kc=kc, vc=vc, tables=t.to(torch.int32).numpy(),
                slots=np.array(slots, np.int32), lens=w.context_lens[seqs].numpy(),
                bytes=store_bytes(n_seq, w.Hkv, w.D) + _sample_decode_bytes(w, seqs),
                tokens=int(w.context_lens[seqs].sum()))


def _sample_decode_bytes(w, seqs):
    toks = int(w.context_lens[seqs].sum())
    n = len(seqs)
    return (toks * w.Hkv * w.D * BF16 * 2 + 2 * n * w.Hq * w.D * BF16 + n * w.Hq * 4 +
            sum(-(-int(w.context_lens[s]) // w.block_size) for s in seqs) * 4 + n * 4)


def oracle_step(s, scale, nthreads=0):
    import oracle
    kc, vc = s["kc"].copy(), s["vc"].copy()
    oracle.store(s["k"], s["v"], kc, vc, s["slots"])
    oracle.decode(s["q"], kc, vc, s["tables"], s["lens"], scale, nthreads=nthreads)


def time_oracle_single_core(dev, budget_s: float = 2.0):
    """The oracle on one thread: tiny-decode whole, decode-b64 on its first 4
    sequences; store + decode GB/s of each sample."""
    res = {}
    for cfg, n_seq in ((1, None), (2, 4)):
        w = W.config_workload(cfg, pool_device=dev)
        s = oracle_sample(w, n_seq or w.B)
        t0 = time.perf_counter()
        oracle_step(s, w.scale, nthreads=1)
        one = time.perf_counter() - t0
        reps = max(1, int(budget_s / max(one, 1e-4)))
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle_step(s, w.scale, nthreads=1)
        el = time.perf_counter() - t0
        res[w.name] = {"GB/s": round(s["bytes"] * reps / el / 1e9, 4),
                       "kv_tokens_per_s": round(s["tokens"] * reps / el, 1),
                       "sample": f"{n_seq or w.B} of {w.B} sequences, {reps} passes"}
        del w
    return res


def time_oracle(w, budget_s: float = 12.0, n_seq: int = None):
    """Oracle store+decode on a bounded sample: whole batch repeated until about
    budget_s seconds of CPU work, or fewer sequences if one pass is too long."""
    import oracle
    threads = oracle.hardware_threads()
    if n_seq is None:
        n_seq = w.B
    s = oracle_sample(w, n_seq)
    t0 = time.perf_counter()
    oracle_step(s, w.scale)
    one = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(s, w.scale)
    el = time.perf_counter() - t0
    gbs = s["bytes"] * reps / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "kv_tokens_per_s": round(s["tokens"] * reps / el, 1),
            "sample": f"{n_seq} of {w.B} sequences of the same workload (store + decode), "
                      f"{reps} passes, {el:.1f} s, fp64, {threads} threads"}


# ----------------------------------------------------------------------------
# GPU arm


def _decode_step(pkv, w, dev_inputs, r, ws, out, lse, stream):
    """One step: store of the new tokens and decode, in one launch."""
    q, kn, vn, kc, vc, tables, slots, lens = dev_inputs
    pkv.paged_decode_attention_store(q, kn, vn, slots[r], kc, vc, tables[r], lens, w.scale,
                                     out=out, lse=lse, workspace=ws, stream=stream)


def _decode_step_two_calls(pkv, w, dev_inputs, r, ws, out, lse, stream):
    """The same step as kv_cache_store followed by paged_decode_attention."""
    q, kn, vn, kc, vc, tables, slots, lens = dev_inputs
    pkv.kv_cache_store(kn, vn, kc, vc, slots[r], stream=stream)
    pkv.paged_decode_attention(q, kc, vc, tables[r], lens, w.scale, out=out, lse=lse,
                               workspace=ws, stream=stream)


def run_gpu(args, world, rank):
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm_peak, _, peak_kind = _peaks()
    if args.profile:
        # same decode-b64 batch, one rotation, pool trimmed to the blocks it
        # uses (~560 MB of K/V on the device): a small case for ncu captures
        w = _trimmed_decode_b64(dev)
    else:
        w = W.config_workload(2, pool_device=dev, rotations=ROTATIONS)
    tables_h = [w.block_tables] + w.extra_tables
    slots_h = [w.slot_mapping] + w.extra_slots
    R = len(tables_h)
    q = w.q.to(dev)
    kn, vn = w.k_new.to(dev), w.v_new.to(dev)
    kc, vc = w.k_cache, w.v_cache
    tables = [t.to(dev) for t in tables_h]
    slots = [s.to(dev) for s in slots_h]
    lens = w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, tables[0].shape[1])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    dev_inputs = (q, kn, vn, kc, vc, tables, slots, lens)

    step_bytes = store_bytes(w.B, w.Hkv, w.D) + decode_bytes(w)

    # The clock sampler starts before the warm-up, so that the warm-up steps
    # run right before the timed region and the GPU does not sit idle first.
    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
    for i in range(args.warmup):
        _decode_step(pkv, w, dev_inputs, i % R, ws, out, lse, stream)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    K = args.steps
    # A step is one launch (store + decode), so the launches run back to back
    # and their average duration is the timed region over K: no event sits
    # between two launches to stretch the step.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        _decode_step(pkv, w, dev_inputs, i % R, ws, out, lse, stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    elapsed_ms = start.elapsed_time(end)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    dec_avg_ms = start.elapsed_time(end) / K   # this rank's own launches
    assert pkv.get_device_error() == pkv.PKV_OK

    value = step_bytes * K * world / (elapsed_ms / 1e3) / 1e9
    kv_tps = w.kv_tokens * K * world / (elapsed_ms / 1e3)
    # the step's one kernel: the new tokens' store and the decode
    dec_gbs = step_bytes / (dec_avg_ms / 1e3) / 1e9

    # for comparison: the same steps as two launches (store, then decode)
    for i in range(3):
        _decode_step_two_calls(pkv, w, dev_inputs, i % R, ws, out, lse, stream)
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a2.record(stream)
    for i in range(K):
        _decode_step_two_calls(pkv, w, dev_inputs, i % R, ws, out, lse, stream)
    b2.record(stream)
    torch.cuda.synchronize()
    two_ms = a2.elapsed_time(b2) / K
    assert pkv.get_device_error() == pkv.PKV_OK

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled 2048-block pool)",
        "config": bench_config(w, world, R),
        "kv_tokens_per_s": round(kv_tps, 1),
        "pct_of_peak_hbm": round(100 * value / hbm_peak, 2),
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel (bf16, producer warp, store fused)",
                     "achieved": round(dec_gbs, 1), "peak": hbm_peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                     "frac": round(dec_gbs / hbm_peak, 4),
                     "traffic": _traffic("decode-b64", step_bytes),
                     "algorithmic_bytes_per_launch": step_bytes,
                     "avg_launch_us": round(dec_avg_ms * 1e3, 2)},
        "two_launch_step": {"ms_per_step": round(two_ms, 5),
                            "value": round(step_bytes / (two_ms / 1e3) / 1e9, 2),
                            "note": "kv_cache_store + paged_decode_attention"},
        "clocks": clk,
    }
    if rank == 0 and not args.profile:
        result["e2e"] = run_e2e(pkv, w, dev_inputs, ws, stream, K, step_bytes)
        if not args.no_extras:
            del dev_inputs, kc, vc, tables, slots, ws, out, lse
            w = None
            torch.cuda.empty_cache()
            result["extras"] = run_extras(pkv, dev, hbm_peak, args)
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = time_oracle(W.config_workload(2, pool_device=dev))
            result["cpu_baseline"]["single_core"] = time_oracle_single_core(dev)
    return result


def bench_config(w, world, rotations=ROTATIONS):
    """The workload description both arms print (the same dict for the same
    workload)."""
    return {"workload": WORKLOAD, "global_batch": w.B * world,
            "kv_tokens_per_step": w.kv_tokens, "store_tokens_per_step": w.B,
            "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {decode_bytes(w) / 1e6:.0f} MB K/V per step, "
                  f"{rotations} rotating batches with disjoint blocks"}


def _trimmed_decode_b64(dev):
    lens = W._uniform_ints(512, 4096, 64, W.seed_for(2))
    nblk = sum(-(-x // W.BLOCK_SIZE) for x in lens)
    return W.make_decode(lens, 16, 8, nblk, W.seed_for(2), name="decode-b64",
                         pool_device=dev)


def run_e2e(pkv, w, dev_inputs, ws, stream, K, step_bytes):
    """Same steps through the public API with each step's inputs in pinned host
    memory: every step copies q, new K/V, slots, tables and lengths host to
    device, runs the fused store + decode and copies out and lse back, all
    inside the timed region.  As in a serving loop, the copies run on a second
    stream and overlap the neighbouring steps' kernels: two sets of device
    input and output buffers, ordered by events (step i's inputs land before
    its kernel; its buffers are refilled only after its kernel and its
    read-back are done)."""
    q, kn, vn, kc, vc, tables, slots, lens = dev_inputs
    R = len(tables)
    h_q = w.q.pin_memory()
    h_k, h_v = w.k_new.pin_memory(), w.v_new.pin_memory()
    h_tables = [t.cpu().pin_memory() for t in tables]
    h_slots = [s.cpu().pin_memory() for s in slots]
    h_lens = w.context_lens.pin_memory()
    h_out = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(2)]
    h_lse = [torch.empty((w.B, w.Hq), dtype=torch.float32).pin_memory() for _ in range(2)]
    bufs = [dict(tab=torch.empty_like(tables[0]), slot=torch.empty_like(slots[0]),
                 q=torch.empty_like(q), k=torch.empty_like(kn), v=torch.empty_like(vn),
                 lens=torch.empty_like(lens), out=torch.empty_like(q),
                 lse=torch.empty((w.B, w.Hq), dtype=torch.float32, device=q.device))
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_tables[0], h_slots[0],
                                                      h_lens))
    d2h = h_out[0].numel() * h_out[0].element_size() + h_lse[0].numel() * 4
    copy = torch.cuda.Stream(device=q.device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    landed = [ev(), ev()]    # inputs of the set copied in
    computed = [ev(), ev()]  # kernel of the set done
    returned = [ev(), ev()]  # results of the set copied out
    for e in returned:
        e.record(copy)

    def copy_in(i):  # step i's inputs into set i & 1, once that set's last step is done
        j, r = i & 1, i % R
        bf = bufs[j]
        with torch.cuda.stream(copy):
            copy.wait_event(returned[j])
            bf["q"].copy_(h_q, non_blocking=True)
            bf["k"].copy_(h_k, non_blocking=True)
            bf["v"].copy_(h_v, non_blocking=True)
            bf["tab"].copy_(h_tables[r], non_blocking=True)
            bf["slot"].copy_(h_slots[r], non_blocking=True)
            bf["lens"].copy_(h_lens, non_blocking=True)
            landed[j].record(copy)

    def launch(i):
        j = i & 1
        bf = bufs[j]
        stream.wait_event(landed[j])
        pkv.paged_decode_attention_store(bf["q"], bf["k"], bf["v"], bf["slot"], kc, vc,
                                         bf["tab"], bf["lens"], w.scale, out=bf["out"],
                                         lse=bf["lse"], workspace=ws, stream=stream)
        computed[j].record(stream)

    def copy_out(i):
        j = i & 1
        with torch.cuda.stream(copy):
            copy.wait_event(computed[j])
            h_out[j].copy_(bufs[j]["out"], non_blocking=True)
            h_lse[j].copy_(bufs[j]["lse"], non_blocking=True)
            returned[j].record(copy)

    def run(n):
        # the copy stream takes step i+1's inputs before step i's results, so
        # the inputs land while step i's kernel runs
        copy_in(0)
        for i in range(n):
            launch(i)
            if i + 1 < n:
                copy_in(i + 1)
            copy_out(i)

    run(4)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy.wait_stream(stream)
    run(K)
    stream.wait_stream(copy)   # the last read-back is inside the timed region
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": round(step_bytes * K / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / K, 5),
            "note": "pinned host buffers; H2D, fused kernel and D2H of every step inside "
                    "the timed region, copies on a second stream overlapping the "
                    "neighbouring steps' kernels"}


def _time_calls(fn, reps, stream):
    """Median and min per-call device time (CUDA events around each call)."""
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = [x.elapsed_time(y) for x, y in times]
    return statistics.median(ms), min(ms)


def _flush_l2(buf):
    buf.add_(1)


def run_extras(pkv, dev, hbm_peak, args):
    """The other workloads: decode GB/s on tiny / prefix-shared / long contexts
    (L2 flushed before each timed call), the tiny one also under CUDA-graph
    replay, and chunked-prefill TFLOP/s plus its store."""
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    res = {}
    for cfg in (1, 3, 5):
        w = W.config_workload(cfg, pool_device=dev)
        q, kc, vc = w.q.to(dev), w.k_cache, w.v_cache
        tables, lens = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, tables.shape[1])
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)

        def call():
            pkv.paged_decode_attention(q, kc, vc, tables, lens, w.scale, out=out, lse=lse,
                                       workspace=ws, stream=stream)
        for _ in range(10):
            call()
        times = []
        for _ in range(50):
            _flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        ms = sorted(x.elapsed_time(y) for x, y in times)
        med = ms[len(ms) // 2]
        entry = {"workload": w.name, "median_us": round(med * 1e3, 2),
                 "min_us": round(ms[0] * 1e3, 2), "kv_tokens": w.kv_tokens,
                 "kv_tokens_per_s": round(w.kv_tokens / (med / 1e3), 1),
                 "splits": pkv.paged_decode_num_splits(w.B, w.Hq, w.Hkv, w.D, tables.shape[1])}
        gbs = decode_bytes(w) / (med / 1e3) / 1e9
        entry["GB/s"] = round(gbs, 1)
        entry["frac_of_peak"] = round(gbs / hbm_peak, 4)
        if cfg == 3:
            ub = decode_bytes(w, unique=True) / (med / 1e3) / 1e9
            entry["unique_GB/s"] = round(ub, 1)
            entry["unique_frac_of_peak"] = round(ub / hbm_peak, 4)
            entry["note"] = ("GB/s counts the shared prefix once per sequence (logical); "
                             "unique_GB/s counts it once")
            # the same batch through the shared-prefix entry point
            P = w.shared_prefix_blocks * w.block_size
            need = pkv.paged_decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D,
                                                                  tables.shape[1], P)
            ws2 = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)

            def call_sp():
                pkv.paged_decode_attention_shared_prefix(q, kc, vc, tables, lens, w.scale, P,
                                                         out=out, lse=lse, workspace=ws2,
                                                         stream=stream)
            for _ in range(10):
                call_sp()
            times = []
            for _ in range(50):
                _flush_l2(flush)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call_sp()
                b.record(stream)
                times.append((a, b))
            torch.cuda.synchronize()
            ms2 = sorted(x.elapsed_time(y) for x, y in times)
            med2 = ms2[len(ms2) // 2]
            ub2 = decode_bytes(w, unique=True) / (med2 / 1e3) / 1e9
            entry["shared_prefix_path"] = {
                "median_us": round(med2 * 1e3, 2), "min_us": round(ms2[0] * 1e3, 2),
                "unique_GB/s": round(ub2, 1), "unique_frac_of_peak": round(ub2 / hbm_peak, 4),
                "kv_tokens_per_s": round(w.kv_tokens / (med2 / 1e3), 1),
                "note": "paged_decode_attention_shared_prefix: the 2048-token prefix "
                        "attended once per kv head on tcgen05, then split decode of the "
                        "private suffixes"}
            del ws2
        if cfg == 1:
            g = torch.cuda.CUDAGraph()
            s2 = torch.cuda.Stream()
            s2.wait_stream(stream)
            with torch.cuda.stream(s2):
                call_g = lambda: pkv.paged_decode_attention(  # noqa: E731
                    q, kc, vc, tables, lens, w.scale, out=out, lse=lse, workspace=ws, stream=s2)
                call_g()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s2):
                    for _ in range(64):
                        call_g()
            stream.wait_stream(s2)
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(10):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            per = a.elapsed_time(b) / 640
            entry["graph_replay_us_per_call"] = round(per * 1e3, 2)
            entry["graph_replay_GB/s"] = round(decode_bytes(w) / (per / 1e3) / 1e9, 1)
            # the same with PKV_DECODE_METADATA_READY: tables and lengths are
            # written before the graph and never by a kernel in it
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s2):
                call_m = lambda: pkv.paged_decode_attention(  # noqa: E731
                    q, kc, vc, tables, lens, w.scale, out=out, lse=lse, workspace=ws, stream=s2,
                    metadata_ready=True)
                call_m()
                torch.cuda.synchronize()
                with torch.cuda.graph(g2, stream=s2):
                    for _ in range(64):
                        call_m()
            stream.wait_stream(s2)
            g2.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(10):
                g2.replay()
            b.record(stream)
            torch.cuda.synchronize()
            assert pkv.get_device_error() == pkv.PKV_OK
            per_m = a.elapsed_time(b) / 640
            entry["graph_replay_metadata_ready_us_per_call"] = round(per_m * 1e3, 2)
            # the bucketed graph runner: one graph launch (pad, fused store +
            # decode) per call from the host, 64 calls back to back
            from paged_kv_cache_214_gb300 import graphs
            runner = graphs.DecodeGraphs(kc, vc, w.Hq, tables.shape[1], 8, w.scale)
            runner.step(q, w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev), tables,
                        lens, stream=stream)
            for _ in range(10):
                runner.run(w.B, stream=stream)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(64):
                runner.run(w.B, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            assert pkv.get_device_error() == pkv.PKV_OK
            per_r = a.elapsed_time(b) / 64
            entry["graph_runner_us_per_call"] = round(per_r * 1e3, 2)
            entry["graph_runner_bucket"] = runner.bucket_for(w.B)
            runner.close()
            entry["note"] = "launch-latency bound: 4.45 MB of K/V per call"
        res[w.name] = entry
        del w, q, kc, vc, tables, lens, out, lse, ws
        torch.cuda.empty_cache()
    # chunked prefill: store of 8192 new tokens, then prefill attention
    w = W.config_workload(4, pool_device=dev)
    q, kc, vc = w.q.to(dev), w.k_cache, w.v_cache
    kn, vn, slots = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
    tables, cq, ck = w.block_tables.to(dev), w.cu_seqlens_q.to(dev), w.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device=dev)
    entry = {"workload": w.name}
    st_med, _ = _time_calls(lambda: pkv.kv_cache_store(kn, vn, kc, vc, slots, stream=stream),
                            50, stream)
    sb = store_bytes(q.shape[0], w.Hkv, w.D)
    entry["store_us"] = round(st_med * 1e3, 2)
    entry["store_GB/s"] = round(sb / (st_med / 1e3) / 1e9, 1)
    try:
        def pcall():
            pkv.paged_prefill_attention(q, kc, vc, tables, cq, ck, w.max_seqlen_q,
                                        w.max_seqlen_k, w.scale, out=out, lse=lse, stream=stream)
        for _ in range(10):
            pcall()
        med, mn = _time_calls(pcall, 50, stream)
        fl = prefill_flops(w)
        _, bf16_peak, kind = _peaks()
        entry.update({"prefill_us": round(med * 1e3, 2), "prefill_min_us": round(mn * 1e3, 2),
                      "flop": fl, "TFLOP/s": round(fl / (med / 1e3) / 1e12, 1),
                      "frac_of_bf16_peak": round(fl / (med / 1e3) / 1e12 / bf16_peak, 4),
                      "peak_kind": f"{kind} bf16_tflops"})
    except Exception as e:  # reported, not hidden
        entry["prefill_error"] = str(e)
    res[w.name] = entry
    del w, q, kc, vc, kn, vn, slots, tables, cq, ck, out, lse
    torch.cuda.empty_cache()
    res["verify-b64-q4"] = run_verify_extra(pkv, dev, hbm_peak, flush, stream)
    for cfg in (2, 5):
        e = run_fp8_extra(pkv, dev, hbm_peak, flush, stream, cfg)
        res[e["workload"]] = e
    return res


def run_fp8_extra(pkv, dev, hbm_peak, flush, stream, cfg):
    """Decode over the FP8 (E4M3) cache: the bf16 pool of a decode workload is
    quantized once with kv_cache_store_fp8 (per-tensor scales), then
    paged_decode_attention_fp8 is timed with L2 flushed before each call."""
    w = W.config_workload(cfg, pool_device=dev)
    NB, bs = w.num_blocks, w.block_size
    k8 = torch.empty((NB, bs, w.Hkv, w.D), dtype=torch.uint8, device=dev)
    v8 = torch.empty_like(k8)
    ks, vs = 6.0 / 448, 6.0 / 448
    every = torch.arange(NB * bs, dtype=torch.int32, device=dev)
    pkv.kv_cache_store_fp8(w.k_cache.view(-1, w.Hkv, w.D), w.v_cache.view(-1, w.Hkv, w.D),
                           k8, v8, every, ks, vs, stream=stream)
    del every
    w.k_cache = w.v_cache = None
    torch.cuda.empty_cache()
    q = w.q.to(dev)
    tables, lens = w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, tables.shape[1])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)

    def call():
        pkv.paged_decode_attention_fp8(q, k8, v8, tables, lens, w.scale, ks, vs, out=out,
                                       lse=lse, workspace=ws, stream=stream)
    kn, vn, slots = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)

    def fused():
        pkv.paged_decode_attention_fp8_store(q, kn, vn, slots, k8, v8, tables, lens, w.scale,
                                             ks, vs, out=out, lse=lse, workspace=ws,
                                             stream=stream)

    def median_us(fn):
        for _ in range(10):
            fn()
        times = []
        for _ in range(50):
            _flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        ms = sorted(x.elapsed_time(y) for x, y in times)
        return ms[len(ms) // 2], ms[0]
    med, mn = median_us(call)
    med_f, _ = median_us(fused)
    gbs = decode_bytes(w, kv_elem_bytes=1) / (med / 1e3) / 1e9
    entry = {"workload": w.name + "-fp8", "median_us": round(med * 1e3, 2),
             "min_us": round(mn * 1e3, 2), "kv_tokens": w.kv_tokens,
             "kv_tokens_per_s": round(w.kv_tokens / (med / 1e3), 1), "GB/s": round(gbs, 1),
             "frac_of_peak": round(gbs / hbm_peak, 4),
             "fused_store_step_us": round(med_f * 1e3, 2),
             "note": "E4M3 K/V, one byte per element (GB/s counts those bytes); "
                     "fused_store_step_us: the step's store of the new tokens and the "
                     "decode as one launch (paged_decode_attention_fp8_store)"}
    del w, q, k8, v8, tables, lens, out, lse, ws, kn, vn, slots
    torch.cuda.empty_cache()
    return entry


def run_verify_extra(pkv, dev, hbm_peak, flush, stream):
    """Speculative verify: the decode-b64 batch with 4 proposed tokens per
    sequence (q_len = 4), through the multi-query decode and, for comparison,
    through the 128-row tcgen05 prefill on the same inputs.  L2 flushed before
    each timed call."""
    qn = 4
    lens = W._uniform_ints(512, 4096, 64, W.seed_for(2))
    w = W.make_prefill([L - qn for L in lens], [qn] * len(lens), 16, 8, 2048,
                       W.seed_for(2) + 1, name="verify-b64-q4", pool_device=dev)
    q = w.q.to(dev)
    kc, vc = w.k_cache, w.v_cache
    tables, cq, ck = w.block_tables.to(dev), w.cu_seqlens_q.to(dev), w.cu_seqlens_k.to(dev)
    ctx = torch.tensor(w.k_lens, dtype=torch.int32, device=dev)
    q4 = q.view(w.B, qn, w.Hq, w.D)
    out, lse = torch.empty_like(q4), torch.empty((w.B, qn, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_multiquery_workspace_bytes(w.B, qn, w.Hq, w.Hkv, w.D, tables.shape[1])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(10):
            fn()
        times = []
        for _ in range(50):
            _flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        ms = sorted(x.elapsed_time(y) for x, y in times)
        return ms[len(ms) // 2]

    med = timed(lambda: pkv.paged_decode_attention_multiquery(
        q4, kc, vc, tables, ctx, w.scale, out=out, lse=lse, workspace=ws, stream=stream))
    kv_tokens = int(sum(w.k_lens))
    nbytes = kv_tokens * w.Hkv * w.D * 2 * 2 + 2 * q.numel() * 2 + lse.numel() * 4
    out2 = torch.empty_like(q)
    lse2 = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device=dev)
    med_p = timed(lambda: pkv.paged_prefill_attention(
        q, kc, vc, tables, cq, ck, w.max_seqlen_q, w.max_seqlen_k, w.scale, out=out2, lse=lse2,
        stream=stream))
    gbs = nbytes / (med / 1e3) / 1e9
    return {"workload": w.name, "q_len": qn, "median_us": round(med * 1e3, 2),
            "kv_tokens": kv_tokens, "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
            "verified_tokens_per_s": round(w.B * qn / (med / 1e3), 1),
            "prefill_path_us": round(med_p * 1e3, 2),
            "note": "paged_decode_attention_multiquery: 8 (position, head) rows per kv head, "
                    "all in one split-K decode block (K/V read once per kv head); "
                    "prefill_path_us: the same batch through paged_prefill_attention (one "
                    "tile per query head)"}


def _traffic(workload: str, algorithmic: int):
    """DRAM bytes per launch from the committed ncu summary of the same kernel
    source, or None if the kernel changed since the counters were taken."""
    import hashlib
    path = os.path.join(_ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[workload]
        src = open(os.path.join(_ROOT, "paged_kv_cache_214_gb300", "csrc",
                                rec["source"])).read().encode()
        if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha"]:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = W.config_workload(2, pool_device=dev)
    threads = oracle.hardware_threads()
    # size each step so that warmup + steps finish within about two minutes
    probe = oracle_sample(w, 1)
    t0 = time.perf_counter()
    oracle_step(probe, w.scale)
    per_seq = max(time.perf_counter() - t0, 1e-3)
    per_step_budget = min(2.0, 120.0 / max(args.steps + args.warmup, 1))
    n_seq = int(max(1, min(w.B, per_step_budget / per_seq)))
    s = oracle_sample(w, n_seq)
    for _ in range(args.warmup):
        oracle_step(s, w.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(s, w.scale)
    el = time.perf_counter() - t0
    value = s["bytes"] * args.steps / el / 1e9
    sample = (f"{n_seq} of {w.B} sequences of the decode-b64 workload per step "
              f"(store + decode, fp64)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "kv_tokens_per_s": round(s["tokens"] * args.steps / el, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_prefill_profile(args):
    """Small-footprint prefill run for ncu: chunked-prefill-b16 (store of the
    8192 new tokens, then prefill), warmup + steps calls, one JSON line."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    # chunked-prefill-b16 shapes with the pool trimmed to the 96 blocks it uses
    w = W.make_prefill([1024] * 16, [512] * 16, 32, 8, 96, W.seed_for(4),
                       name="chunked-prefill-b16", pool_device=dev)
    q, kc, vc = w.q.to(dev), w.k_cache, w.v_cache
    kn, vn, slots = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
    tables, cq, ck = w.block_tables.to(dev), w.cu_seqlens_q.to(dev), w.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    pkv.kv_cache_store(kn, vn, kc, vc, slots, stream=stream)

    def call():
        pkv.paged_prefill_attention(q, kc, vc, tables, cq, ck, w.max_seqlen_q, w.max_seqlen_k,
                                    w.scale, out=out, lse=lse, stream=stream)
    for _ in range(args.warmup):
        call()
    med, mn = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    fl = prefill_flops(w)
    print(json.dumps({"workload": w.name, "prefill_us": round(med * 1e3, 2),
                      "TFLOP/s": round(fl / (med / 1e3) / 1e12, 1)}), flush=True)


def run_shared_prefix_profile(args):
    """Small-footprint shared-prefix decode run for ncu: the
    prefix-shared-decode-b256 batch with the pool trimmed to the blocks it
    uses."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    s = W.seed_for(3)
    lens = [2048 + x + 1 for x in W._uniform_ints(0, 6144, 256, s)]
    nblk = 8 + sum(-(-L // W.BLOCK_SIZE) - 8 for L in lens)
    w = W.make_decode(lens, 32, 8, nblk, s, name="prefix-shared-decode-b256",
                      shared_prefix_tokens=2048, store_new_token=False, pool_device=dev)
    q, tables, ctx = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D,
                                                          tables.shape[1], 2048)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        pkv.paged_decode_attention_shared_prefix(q, w.k_cache, w.v_cache, tables, ctx, w.scale,
                                                 2048, out=out, lse=lse, workspace=ws,
                                                 stream=stream)
    for _ in range(args.warmup):
        call()
    med, _ = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    ub = decode_bytes(w, unique=True) / (med / 1e3) / 1e9
    print(json.dumps({"workload": w.name, "us": round(med * 1e3, 2),
                      "unique_GB/s": round(ub, 1)}), flush=True)


def run_fp8_decode_profile(args, long_ctx: bool, fused_store: bool = False):
    """Small-footprint FP8 decode run for ncu: the decode-b64 shapes (2 query
    heads per kv head) or, with `long_ctx`, the first 2 sequences of
    long-decode-b8 (4 query heads per kv head) with the 37 splits the planner
    picks for the full batch, as run_long_decode_profile; pools quantized once
    with kv_cache_store_fp8.
    `fused_store`: the decode-b64 step's store of the new tokens and the decode
    in one launch (paged_decode_attention_fp8_store)."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    if long_ctx:
        lens = W._uniform_ints(32768, 131072, 8, W.seed_for(5))[:2]
        Hq, name, maxblk, splits = 32, "long-decode-b8-fp8-2seq", 512, 37
    else:
        lens = W._uniform_ints(512, 4096, 64, W.seed_for(2))
        Hq, name, maxblk, splits = 16, "decode-b64-fp8", None, 0
    nblk = sum(-(-L // W.BLOCK_SIZE) for L in lens)
    w = W.make_decode(lens, Hq, 8, nblk, W.seed_for(2), name=name,
                      store_new_token=fused_store, pool_device=dev, max_blocks_per_seq=maxblk)
    k8 = torch.empty((nblk, w.block_size, w.Hkv, w.D), dtype=torch.uint8, device=dev)
    v8 = torch.empty_like(k8)
    ks = vs = 6.0 / 448
    every = torch.arange(nblk * w.block_size, dtype=torch.int32, device=dev)
    pkv.kv_cache_store_fp8(w.k_cache.view(-1, w.Hkv, w.D), w.v_cache.view(-1, w.Hkv, w.D),
                           k8, v8, every, ks, vs)
    w.k_cache = w.v_cache = None
    q, tables, ctx = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, tables.shape[1],
                                            num_splits=splits)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    if fused_store:
        kn, vn, slots = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)

        def call():
            pkv.paged_decode_attention_fp8_store(q, kn, vn, slots, k8, v8, tables, ctx, w.scale,
                                                 ks, vs, out=out, lse=lse, workspace=ws,
                                                 num_splits=splits, stream=stream)
    else:
        def call():
            pkv.paged_decode_attention_fp8(q, k8, v8, tables, ctx, w.scale, ks, vs, out=out,
                                           lse=lse, workspace=ws, num_splits=splits,
                                           stream=stream)
    for _ in range(args.warmup):
        call()
    med, _ = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    gbs = decode_bytes(w, kv_elem_bytes=1) / (med / 1e3) / 1e9
    print(json.dumps({"workload": w.name, "us": round(med * 1e3, 2), "GB/s": round(gbs, 1)}),
          flush=True)


def run_long_decode_profile(args):
    """Small-footprint long-context decode run for ncu: the first 2 sequences
    of long-decode-b8 (32k-131k tokens) in a pool trimmed to their blocks,
    with the 37 splits the planner picks for the full 8-sequence batch (the
    split-K path with many splits and the log-sum-exp merge)."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    lens = W._uniform_ints(32768, 131072, 8, W.seed_for(5))[:2]
    nblk = sum(-(-L // W.BLOCK_SIZE) for L in lens)
    w = W.make_decode(lens, 32, 8, nblk, W.seed_for(5), name="long-decode-b8-2seq",
                      store_new_token=False, pool_device=dev, max_blocks_per_seq=512)
    q, tables, ctx = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, tables.shape[1],
                                            num_splits=37)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        pkv.paged_decode_attention(q, w.k_cache, w.v_cache, tables, ctx, w.scale, out=out,
                                   lse=lse, workspace=ws, num_splits=37, stream=stream)
    for _ in range(args.warmup):
        call()
    med, _ = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    gbs = decode_bytes(w) / (med / 1e3) / 1e9
    print(json.dumps({"workload": w.name, "us": round(med * 1e3, 2), "GB/s": round(gbs, 1)}),
          flush=True)


def run_verify_profile(args):
    """Small-footprint speculative-verify run for ncu: verify-b64-q4 (the
    decode-b64 contexts with 4 proposed tokens each) in a pool trimmed to the
    blocks it uses, through paged_decode_attention_multiquery."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    qn = 4
    lens = W._uniform_ints(512, 4096, 64, W.seed_for(2))
    nblk = sum(-(-L // W.BLOCK_SIZE) for L in lens)
    w = W.make_prefill([L - qn for L in lens], [qn] * len(lens), 16, 8, nblk,
                       W.seed_for(2) + 1, name="verify-b64-q4", pool_device=dev)
    q = w.q.to(dev).view(w.B, qn, w.Hq, w.D)
    tables = w.block_tables.to(dev)
    ctx = torch.tensor(w.k_lens, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, qn, w.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_multiquery_workspace_bytes(w.B, qn, w.Hq, w.Hkv, w.D,
                                                       tables.shape[1])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        pkv.paged_decode_attention_multiquery(q, w.k_cache, w.v_cache, tables, ctx, w.scale,
                                              out=out, lse=lse, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        call()
    med, _ = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    print(json.dumps({"workload": w.name, "us": round(med * 1e3, 2)}), flush=True)


def run_tiny_profile(args):
    """tiny-decode for ncu: the 4-sequence decode (one split per sequence)."""
    from paged_kv_cache_214_gb300 import pkv
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.config_workload(1, pool_device=dev)
    q, tables, ctx = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        pkv.paged_decode_attention(q, w.k_cache, w.v_cache, tables, ctx, w.scale, out=out,
                                   lse=lse, stream=stream)
    for _ in range(args.warmup):
        call()
    med, _ = _time_calls(call, args.steps, stream)
    assert pkv.get_device_error() == pkv.PKV_OK
    print(json.dumps({"workload": w.name, "us": round(med * 1e3, 2)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-kernel", default="decode",
                    choices=["decode", "prefill", "shared-prefix", "fp8-decode",
                             "fp8-decode-store", "fp8-decode-long", "long-decode", "verify",
                             "tiny"],
                    help="with --profile: which kernel the run exercises")
    ap.add_argument("--profile", action="store_true",
                    help="small-footprint run for ncu: one batch, trimmed pool, "
                         "no extras / e2e / CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        args.no_extras = True
        args.no_cpu_baseline = True
    world, rank, local = dist_setup(args)
    if args.profile_kernel == "prefill":
        run_prefill_profile(args)
        return
    if args.profile_kernel == "shared-prefix":
        run_shared_prefix_profile(args)
        return
    if args.profile_kernel in ("fp8-decode", "fp8-decode-long", "fp8-decode-store"):
        run_fp8_decode_profile(args, args.profile_kernel == "fp8-decode-long",
                               fused_store=args.profile_kernel == "fp8-decode-store")
        return
    if args.profile_kernel == "long-decode":
        run_long_decode_profile(args)
        return
    if args.profile_kernel == "verify":
        run_verify_profile(args)
        return
    if args.profile_kernel == "tiny":
        run_tiny_profile(args)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_gpu(args, world, rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
