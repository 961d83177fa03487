"""Benchmark of one paged decode step on GB300.

A step is one pass of the device path over one batch: kv_append of one new
token per sequence into its slot, then paged decode attention over every
sequence's context (split-context reduction included when the context is
partitioned).  Copy-on-write (block_copy) is part of the path but this batch
shares no blocks, so its step has no pairs to copy.

Workload (default): an OPT-13B-shaped attention layer — 40 heads of 128 (MHA),
fp16, blocks of 16 tokens, 64 sequences with lognormal context lengths
(median 500, sigma 1, clipped to [16, 2048]) whose blocks are shuffled
through a pool 1.3x the size needed; q/K/V ~ N(0, 1), seeded.  Each step
rewrites the token at the last position (the step's new token) and attends
over the whole context, so every step does the same work.

Prints one JSON line: value = algorithmic HBM bytes of the step / step time
(GB/s, summed over ranks), plus decode seqs/s, the roofline of the decode
call, an end-to-end figure through the C ABI with host buffers, the oracle
timed on host cores, and SM clocks sampled during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention HBM GB/s (% of GB300 peak) and decode seqs/s per layer"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="opt13b",
                    choices=["opt13b", "gqa4k", "prefill", "prefill_shapes", "sweep", "shared",
                             "groups"])
    ap.add_argument("--decode-path", type=int, default=0, choices=[0, 1, 2],
                    help="decode kernel: 0 = the library's choice, 1 = CUDA cores, "
                         "2 = tensor cores where supported")
    ap.add_argument("--only", default=None,
                    help="--workload sweep: one case as block_size,batch,ctx; --workload "
                         "prefill_shapes: one case's index (for profiler captures)")
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128],
                    help="--workload groups: head size")
    ap.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32, 64, 128],
                    help="--workload groups: tokens per block")
    ap.add_argument("--group", type=int, default=0,
                    help="one query-head group size for --workload groups (0 = all)")
    ap.add_argument("--partition", type=int, default=0, help="tokens per partition (0 = library)")
    ap.add_argument("--path", default="fused", choices=["fused", "separate"],
                    help="one fused append+decode launch, or kv_append then decode")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-buffers", type=int, default=2,
                    help="staging buffers of the end-to-end loop (inputs copied that many - 1 "
                         "steps ahead)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="fewer sequences than the workload's (for profiler captures)")
    return ap.parse_args()


# ------------------------------------------------------------- utilities --

def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_247_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


DECODE_SOURCES = ("decode.cu", "common.cuh", "overlap.cuh")
DECODE_TC_SOURCES = ("decode_tc.cu", "decode.cu", "common.cuh", "overlap.cuh", "tcgen05.cuh")
PREFILL_SOURCES = ("prefill.cu", "common.cuh", "tcgen05.cuh")


def ncu_traffic(kernel_key, workload, sources=DECODE_SOURCES):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[workload][kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != source_hash(*sources):
        return None
    return rec.get("dram_bytes_per_launch")


def set_decode_path(args):
    """Apply --decode-path (process-wide in the library)."""
    from paged_kv_cache_247_gb300 import _lib
    _lib.check(_lib.load().pkv_set_decode_path(args.decode_path), "pkv_set_decode_path")


def max_over_ranks(ms, world):
    """The slowest rank's time: every rank returns the same value (gloo or
    NCCL all-reduce MAX; a no-op on one rank)."""
    t = torch.tensor([float(ms)], dtype=torch.float64)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi sampling every 100 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- workload --

def make_workload(name, device, num_seqs=None):
    from paged_kv_cache_247_gb300 import workloads as W
    if name == "opt13b":
        case = W.opt13b_layer_decode(device=device, num_seqs=num_seqs)
        desc = dict(W.OPT13B_LAYER)
        label = "OPT-13B-shaped layer decode + kv_append"
    else:
        case = W.gqa_4k_decode(device=device, num_seqs=num_seqs)
        desc = dict(W.GQA_4K)
        label = "GQA 32q/8kv decode, ctx 4096 + kv_append"
    S, Hq, D = case.q.shape
    Hkv = case.k_cache.shape[1]
    k_new, v_new = W.new_tokens(11, S, Hkv, D, desc["dtype"], device=device)
    slots = W.last_position_slots(case).to(device)
    return case, k_new, v_new, slots, desc, label


def step_bytes(case):
    """Algorithmic HBM bytes of one step: decode reads each context's K and V
    once plus q, the table and the lengths, and writes out; the append reads
    and writes one K and one V row per sequence (plus its slot)."""
    S, Hq, D = case.q.shape
    Hkv, B = case.k_cache.shape[1], case.block_size
    e = case.q.element_size()
    lens = case.context_lens.cpu().numpy().astype(np.int64)
    kv = int(lens.sum()) * 2 * Hkv * D * e
    decode = kv + 2 * S * Hq * D * e + int((-(-lens // B)).sum()) * 4 + S * 4
    append = 2 * 2 * S * Hkv * D * e + S * 8
    return decode, append


def contiguous_baseline(pkv, case, out, part, dev, stream, iters):
    """Paged vs contiguous decode on the same tokens, both on the CUDA-core
    kernel (the contiguous layout has only that one), at the same partition:
    the ratio of the two times is the cost of the indirection."""
    S, Hq, D = case.q.shape
    Hkv, B = case.k_cache.shape[1], case.block_size
    cap = case.max_context_len
    kc = torch.zeros((S, Hkv, cap, D), dtype=case.q.dtype, device=dev)
    vc = torch.zeros_like(kc)
    tables = case.block_tables.long()
    for s, n in enumerate(case.context_lens.tolist()):
        nb = -(-n // B)
        ids = tables[s, :nb]
        kc[s, :, :n] = case.k_cache[ids].permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :n]
        vc[s, :, :n] = case.v_cache[ids].permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :n]
    ws = torch.empty(max(16, pkv.decode_workspace_size(S, Hq, Hkv, D, cap, part)),
                     dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        return timed_steps(fn, iters, stream, 0.05) / iters

    path = pkv.load_library().pkv_get_decode_path()
    pkv.set_decode_path(1)
    try:
        t_paged = timed(lambda: pkv.paged_attn_decode(
            out, case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
            case.scale, cap, partition_size=part, workspace=ws))
    finally:
        pkv.set_decode_path(path)
    t_contig = timed(lambda: pkv.contiguous_attn_decode(
        out, case.q, kc, vc, case.context_lens, case.scale, partition_size=part, workspace=ws))
    reserved = kc.numel() * kc.element_size() * 2
    held = int(case.context_lens.sum().item()) * Hkv * D * case.q.element_size() * 2
    del kc, vc
    torch.cuda.empty_cache()
    return {"paged_decode_ms": round(t_paged, 5), "contiguous_decode_ms": round(t_contig, 5),
            "indirection_overhead_pct": round(100.0 * (t_paged / t_contig - 1.0), 2),
            "contiguous_reserved_bytes": reserved, "paged_held_bytes": held,
            "partition_size": part, "iters": iters, "kernel": "CUDA-core decode kernel, both"}


def time_alone(fn, flush, stream, iters):
    """Mean device time of fn() in ms, each call timed alone: read `flush`
    (larger than L2; None keeps the cache as it is) to evict the call's data,
    then hold the stream in a bounded device-side wait (about 0.1-0.15 ms) so
    the host has queued the call before the start event fires and its launch
    cost stays out."""
    total = 0.0
    for _ in range(iters):
        if flush is not None:
            flush.sum()
        torch.cuda._sleep(300_000)  # clock cycles
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
    return total / iters


def launch_floor_ms(flush, stream, iters):
    """An empty kernel (a zero-cycle device-side wait) timed like the calls
    of time_alone: the part of a lone call's time that no kernel avoids
    (the launch leaving the queue, the CTAs starting, the end event)."""
    for _ in range(3):
        torch.cuda._sleep(0)
    return time_alone(lambda: torch.cuda._sleep(0), flush, stream, iters)


def pipelined_steps(stream, n_steps, copy_in, compute, copy_out, hold_ms=5.0, nbuf=2):
    """Mean ms per step of a multi-buffered serving loop, on the device
    clock.  copy_in(b) fills input buffer b on a copy stream, compute(b)
    reads input b and writes output b on `stream`, copy_out(b) reads output
    b back on a second copy stream.  Step i + nbuf - 1's inputs go in, and
    step i's output comes out, while the compute stream moves on; each buffer
    is reused only after the step that last touched it is done with it."""
    dev = stream.device
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(nbuf)]
    done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        hold_stream(hold_ms)  # the host queues the first steps before t0 fires
    t0.record(stream)
    s_in.wait_event(t0)
    for k in range(min(nbuf - 1, n_steps)):
        with torch.cuda.stream(s_in):
            copy_in(k)
        in_ready[k].record(s_in)
    for i in range(n_steps):
        b = i % nbuf
        stream.wait_event(in_ready[b])
        if i >= nbuf:
            stream.wait_event(out_done[b])  # step i-nbuf's output has been read back
        with torch.cuda.stream(stream):
            compute(b)
        done[b].record(stream)
        nxt = i + nbuf - 1
        if nxt < n_steps:
            bn = nxt % nbuf
            if nxt >= nbuf:
                s_in.wait_event(done[bn])  # step nxt-nbuf has read that input buffer
            with torch.cuda.stream(s_in):
                copy_in(bn)
            in_ready[bn].record(s_in)
        s_out.wait_event(done[b])
        with torch.cuda.stream(s_out):
            copy_out(b)
        out_done[b].record(s_out)
    stream.wait_event(out_done[(n_steps - 1) % nbuf])
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n_steps


def cache_ops_bench(pkv, case, dev, stream, peak, iters=30, fill_blocks=400, cow_pairs=112):
    """The two cache-maintenance kernels on their large instances, each call
    timed alone with CUDA events after reading a buffer larger than L2:
    a prompt fill (kv_append of fill_blocks whole blocks, block_size tokens
    each, into blocks drawn at random from the pool) and a copy-on-write batch
    (block_copy of cow_pairs distinct source -> destination blocks).  Bytes
    moved = everything read plus everything written."""
    S, Hq, D = case.q.shape
    Hkv, B, NB = case.k_cache.shape[1], case.block_size, case.k_cache.shape[0]
    e = case.q.element_size()
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1234)
    perm = torch.randperm(NB, generator=gen)
    n_fill = min(fill_blocks, NB)
    T = n_fill * B
    slots = (perm[:n_fill, None] * B + torch.arange(B)[None, :]).reshape(-1).to(dev)
    k_new = torch.randn((T, Hkv, D), generator=gen).to(case.q.dtype).to(dev)
    v_new = torch.randn((T, Hkv, D), generator=gen).to(case.q.dtype).to(dev)
    n_cow = min(cow_pairs, NB // 2)
    pairs = torch.stack([perm[:n_cow], perm[n_cow:2 * n_cow]], dim=1).to(torch.int64).to(dev)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    # L2 is flushed by reading 256 MiB (a write would leave dirty lines whose
    # write-back would compete with the timed call for DRAM bandwidth)
    flush = torch.ones(32 << 20, dtype=torch.float64, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        return time_alone(fn, flush, stream, iters)

    pkv.device_status(clear=True)
    t_app = timed(lambda: pkv.kv_append(k_new, v_new, kc, vc, slots))
    t_cow = timed(lambda: pkv.block_copy(kc, vc, pairs))
    # For scale: torch's own device copy of the same number of bytes (one
    # contiguous buffer read and written), timed the same way.
    ref = {}
    for name, nbytes in (("kv_append_prompt_fill", 2 * T * Hkv * D * e),
                         ("block_copy_cow_batch", 2 * n_cow * Hkv * B * D * e)):
        src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        ref[name] = timed(lambda: dst.copy_(src))
        del src, dst
    # The copy-on-write batch at other sizes, beside torch's copy of the same
    # bytes: how the per-call latency weighs against the bytes moved.
    batches = []
    for n in (28, 224, 448):
        if 2 * n > NB:
            continue
        pr = torch.stack([perm[:n], perm[n:2 * n]], dim=1).to(torch.int64).to(dev)
        t_n = timed(lambda: pkv.block_copy(kc, vc, pr))
        nbytes = 2 * n * Hkv * B * D * e
        src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        t_ref = timed(lambda: dst.copy_(src))
        del src, dst, pr
        gbs = 2 * nbytes / (t_n * 1e-3) / 1e9
        batches.append({"pairs": n, "bytes_moved": 2 * nbytes, "ms": round(t_n, 5),
                        "frac_of_peak": round(gbs / peak, 4),
                        "torch_copy_same_bytes_ms": round(t_ref, 5)})
    floor = launch_floor_ms(flush, stream, iters)
    if pkv.device_status(clear=True) != 0:
        raise RuntimeError("device status flags during the cache-operation bench")
    b_app = 2 * (2 * T * Hkv * D * e)          # K and V rows read, then written
    b_cow = 2 * (2 * n_cow * Hkv * B * D * e)  # K and V blocks read, then written
    del kc, vc, flush
    torch.cuda.empty_cache()

    def rec(ms, nbytes, what, key):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"what": what, "bytes_moved": nbytes, "ms": round(ms, 5), "GB/s": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4),
                "torch_copy_same_bytes_ms": round(ref[key], 5)}

    return {"kv_append_prompt_fill": rec(t_app, b_app, f"{T} tokens x {Hkv} heads into {n_fill} "
                                         "random blocks", "kv_append_prompt_fill"),
            "block_copy_cow_batch": rec(t_cow, b_cow, f"{n_cow} block pairs, K and V",
                                        "block_copy_cow_batch"),
            "block_copy_other_batches": batches,
            "empty_kernel_ms": round(floor, 5),
            "l2": "flushed (256 MiB read) before every timed call",
            "launch": "queued behind a device-side wait, outside the timed region", "iters": iters}


# ------------------------------------------------------------- CPU legs --

def oracle_sample_rate(case, k_new, v_new, slots, seconds, max_seqs=None):
    """Time the fp64 oracle (append + decode) on whole sequences of the
    workload until `seconds` pass; returns (GB/s, sequences done, elapsed)."""
    import oracle
    S, Hq, D = case.q.shape
    Hkv, B = case.k_cache.shape[1], case.block_size
    e = case.q.element_size()
    tables = case.block_tables.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    order = np.random.default_rng(0).permutation(S)
    done, nbytes, t_total = 0, 0, 0.0
    i = 0
    while t_total < seconds and (max_seqs is None or done < max_seqs):
        s = int(order[i % S])
        i += 1
        nb = -(-int(lens[s]) // B)
        ids = torch.from_numpy(tables[s, :nb].astype(np.int64)).to(case.k_cache.device)
        kc = case.k_cache.index_select(0, ids).float().cpu().numpy()
        vc = case.v_cache.index_select(0, ids).float().cpu().numpy()
        q = case.q[s:s + 1].double().cpu().numpy()
        kn = k_new[s:s + 1].float().cpu().numpy()
        vn = v_new[s:s + 1].float().cpu().numpy()
        # the sequence's blocks, relabelled 0..nb-1 in table order
        phys, off = divmod(int(slots[s]), B)
        local_slot = np.array([int(np.nonzero(tables[s, :nb] == phys)[0][0]) * B + off])
        t0 = time.perf_counter()
        kc2, vc2 = oracle.kv_append(kn, vn, kc, vc, local_slot)
        oracle.paged_decode_attention(q, kc2.astype(np.float64), vc2.astype(np.float64),
                                      np.arange(nb)[None, :], [int(lens[s])], case.scale)
        t_total += time.perf_counter() - t0
        done += 1
        nbytes += int(lens[s]) * 2 * Hkv * D * e + 2 * Hq * D * e + 4 * Hkv * D * e
    return nbytes / t_total / 1e9, done, t_total


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def host_info():
    """The host the oracle runs on: CPU model, cores this process may use,
    and the BLAS library numpy calls with its thread count."""
    info = {"cores": cores_used(), "cpu_model": None, "blas": None, "blas_threads": None}
    try:
        with open("/proc/cpuinfo") as f:
            for row in f:
                if row.lower().startswith("model name"):
                    info["cpu_model"] = row.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if info["cpu_model"] is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for row in out.splitlines():
                if row.strip().lower().startswith("model name"):
                    info["cpu_model"] = row.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    if info["cpu_model"] is None:
        import platform
        info["cpu_model"] = platform.machine()
    try:
        from threadpoolctl import threadpool_info
        for lib in threadpool_info():
            if lib.get("user_api") == "blas":
                info["blas"] = f"{lib.get('internal_api')} {lib.get('version')}"
                info["blas_threads"] = lib.get("num_threads")
                break
    except ImportError:
        # No threadpoolctl: ask the OpenBLAS that numpy loaded directly.
        import ctypes
        try:
            with open("/proc/self/maps") as f:
                paths = {row.split()[-1] for row in f if "openblas" in row.lower()}
        except OSError:
            paths = set()
        for path in sorted(paths):
            try:
                so = ctypes.CDLL(path)
            except OSError:
                continue
            for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                         "openblas_get_num_threads"):
                fn = getattr(so, name, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    info["blas"] = "openblas (" + os.path.basename(path) + ")"
                    info["blas_threads"] = int(fn())
                    break
            if info["blas_threads"] is not None:
                break
    return info


def workload_config(case, label, world):
    """The workload as both arms describe it (no execution details)."""
    S, Hq, D = case.q.shape
    decode_b, _ = step_bytes(case)
    return {"workload": label, "num_seqs": S, "num_q_heads": Hq,
            "num_kv_heads": case.k_cache.shape[1], "head_dim": D,
            "block_size": case.block_size,
            "cache_dtype": "fp16" if case.q.dtype == torch.float16 else "bf16",
            "context_tokens": int(case.context_lens.sum().item()),
            "max_context_len": case.max_context_len,
            "l2": f"inputs larger than L2: {decode_b / 1e9:.2f} GB of K/V per step vs 129 MB L2, "
                  "no flush",
            "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ arms --

def run_reference(args, rank, world):
    """The oracle timed on host cores as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    case, k_new, v_new, slots, desc, label = make_workload(args.workload, "cpu", args.num_seqs)
    # bounded so that the whole run stays within a few minutes (at least one
    # whole sequence per step)
    per_step = min(6.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_rate(case, k_new, v_new, slots, per_step / 4, max_seqs=1)
    total_bytes_t, seqs, elapsed = 0.0, 0, 0.0
    for _ in range(args.steps):
        rate, n, t = oracle_sample_rate(case, k_new, v_new, slots, per_step)
        total_bytes_t += rate * t
        seqs += n
        elapsed += t
    value = total_bytes_t / elapsed
    host = host_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * elapsed / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, label, world),
        "decode_seqs_per_s": round(seqs / elapsed, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": host["cores"],
                         "kind": "oracle", "cpu_model": host["cpu_model"], "blas": host["blas"],
                         "blas_threads": host["blas_threads"],
                         "sample": f"{seqs} whole sequences of the workload (append + decode), "
                                   f"random order, ~{per_step:.1f} s per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# SM clock used to turn a bounded device-side wait into cycles: the wait
# lasts at least the requested time at any clock up to the maximum.
MAX_SM_GHZ = 2.07


def hold_stream(ms):
    """Occupy the current stream for about `ms` milliseconds with a bounded
    spin on the device, so that work the host enqueues meanwhile is queued
    before the next event fires."""
    torch.cuda._sleep(int(ms * MAX_SM_GHZ * 1e6))


def queue_ahead_ms(host_ms_per_step, steps):
    """A hold long enough for the host to enqueue the first `steps` steps
    (at most 512 of them: after that the device is already busy)."""
    return min(50.0, 2.0 + 1.5 * host_ms_per_step * min(steps, 512))


def timed_steps(enqueue, K, stream, host_ms):
    """Device time (ms) of K back-to-back steps, measured between two events
    on `stream`.  The stream is first held in a bounded device-side wait while
    the host enqueues the steps, so the start event fires with the steps
    already queued: the host's marshalling of the first launches is not in
    the timed region."""
    torch.cuda.synchronize()
    hold_stream(queue_ahead_ms(host_ms, K))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(K):
        enqueue()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def decode_record(pkv, args, workload, dev, stream, world, K, extras, rank):
    """Time one decode workload: K steps back to back (each: append the new
    token and attend), the kernel's roofline, and the end-to-end figure with
    host buffers.  With `extras` also the other step path, the contiguous
    baseline and the cache-operation kernels."""
    case, k_new, v_new, slots, desc, label = make_workload(workload, dev, args.num_seqs)
    S, Hq, D = case.q.shape
    Hkv = case.k_cache.shape[1]
    e = case.q.element_size()
    out = torch.empty_like(case.q)
    ws_bytes = pkv.decode_workspace_size(S, Hq, Hkv, D, case.max_context_len, args.partition)
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    part = args.partition or pkv.decode_partition_size(S, Hq, Hkv, D, case.max_context_len)
    split = -(-case.max_context_len // part) > 1

    def enqueue(path, qd, kd, vd, sd, td, ld, ev=None, o=None):
        """One step on the stream: append the new token and attend."""
        o = out if o is None else o
        if path == "separate":
            pkv.kv_append(kd, vd, case.k_cache, case.v_cache, sd)
        if ev is not None:
            ev[0].record(stream)
        if path == "separate":
            pkv.paged_attn_decode(o, qd, case.k_cache, case.v_cache, td, ld, case.scale,
                                  case.max_context_len, partition_size=args.partition,
                                  workspace=workspace)
        else:
            pkv.paged_attn_decode_append(o, qd, kd, vd, case.k_cache, case.v_cache, td, ld,
                                         case.scale, case.max_context_len,
                                         partition_size=args.partition, workspace=workspace)
        if ev is not None:
            ev[1].record(stream)

    dev_args = (case.q, k_new, v_new, slots, case.block_tables, case.context_lens)
    launches_per_step = (2 if args.path == "separate" else 1) + (1 if split else 0)

    pkv.device_status(clear=True)
    W = max(3, args.warmup)
    t_host = 0.0
    for i in range(W):
        t0 = time.perf_counter()
        enqueue(args.path, *dev_args)
        if i >= W // 2:
            t_host += time.perf_counter() - t0
    torch.cuda.synchronize()
    host_ms = 1e3 * t_host / (W - W // 2)

    # The separate path's decode launch is sampled with events inside the
    # timed region (at least 10 samples); the fused path has one launch per
    # step, so the timed region itself is the launches' duration.
    ev = {}
    if args.path == "separate":
        every = max(1, min(10, K // 10))
        ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for i in range(0, K, every)}
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    it = iter(range(K))
    elapsed_ms = timed_steps(lambda: enqueue(args.path, *dev_args, ev=ev.get(next(it))),
                             K, stream, host_ms)
    clock_rec = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    flags = pkv.device_status(clear=True)
    if flags:
        raise RuntimeError(f"device status flags {flags} during the bench")
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_step = elapsed_ms / K

    decode_b, append_b = step_bytes(case)
    if args.path == "fused":
        # the fused kernel also writes the new K/V rows (it reads them from
        # the caller instead of the cache: the same bytes)
        kernel_b = decode_b + 2 * S * Hkv * D * e
        kernel_name = "paged_attn_decode_append call (fused append + decode kernel"
        avg_launch_ms = ms_step
        launches_timed = (f"all {K}: the call is the step's only work, so the timed region is "
                          f"{K} back-to-back calls")

        def call_alone():
            enqueue("fused", *dev_args)
    else:
        kernel_b = decode_b
        kernel_name = "paged_attn_decode call (decode kernel"
        samples = [a.elapsed_time(b) for a, b in ev.values()]
        avg_launch_ms = float(np.mean(samples))
        launches_timed = (f"{len(samples)} of {K} steps, events around the decode launch inside "
                          "the timed region")

        def call_alone():
            pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                                  case.context_lens, case.scale, case.max_context_len,
                                  partition_size=args.partition, workspace=workspace)
    kernel_name += " + split reduction)" if split else ")"
    kernel_name += ("; tensor-core kernel paged_decode_tc_kernel" if pkv.decode_uses_tensor_cores(
        S, Hq, Hkv, D, case.max_context_len, args.partition) else "; CUDA-core kernel "
        "paged_decode_kernel")
    # Cross-check: the same call timed alone, launch queued behind a device
    # wait so that it is outside the event pair (K/V larger than L2: no flush).
    alone_ms = time_alone(call_alone, None, stream, max(10, min(K, 50)))
    peak, peak_kind = peak_hbm()
    achieved = kernel_b / (avg_launch_ms * 1e-3) / 1e9
    tc = pkv.decode_uses_tensor_cores(S, Hq, Hkv, D, case.max_context_len, args.partition)
    kname = "paged_decode_tc_kernel" if tc else "paged_decode_kernel"
    traffic = ncu_traffic(f"{kname}:{args.path}", workload,
                          DECODE_TC_SOURCES if tc else DECODE_SOURCES)
    roofline = {"kernel": kernel_name, "bound": "hbm", "achieved": round(achieved, 2),
                "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback",
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": kernel_b, "avg_launch_ms": round(avg_launch_ms, 5),
                "launches_timed": launches_timed,
                "alone_ms": round(alone_ms, 5),
                "alone_frac": round(kernel_b / (alone_ms * 1e-3) / 1e9 / peak, 4),
                "alone_note": "the same call timed alone (launch outside the event pair, no "
                              "overlap with a neighbouring launch)"}
    if avg_launch_ms > ms_step * (1.0 + 1e-6):
        # A launch cannot outlast the step it is part of: the figure is not
        # evidence, so it is not reported.
        roofline = {"rejected": f"average launch {avg_launch_ms:.5f} ms exceeds the step "
                                f"{ms_step:.5f} ms"}

    # End to end through the C ABI with host buffers: every step copies its
    # inputs (q, new K/V, slots, tables, lengths) from pinned host memory and
    # reads the output back.  The step's inputs sit in one pinned staging
    # buffer (each 256-byte aligned), so a step is one host-to-device copy,
    # the launch(es), and one device-to-host copy of the output.  As a
    # serving loop would, the copies run on streams of their own with two
    # staging and two output buffers: step i+1's inputs are copied in and
    # step i's output copied out while the next step computes.  The serial
    # form (copy in, launch, copy out, one after another on one stream) is
    # reported beside it.
    srcs = (("q", case.q), ("k", k_new), ("v", v_new), ("slots", slots),
            ("tables", case.block_tables), ("lens", case.context_lens))
    names = [n for n, _ in srcs]
    offs, total = {}, 0
    for n, x in srcs:
        offs[n] = total
        total += -(-x.numel() * x.element_size() // 256) * 256
    NBUF = max(2, args.e2e_buffers)
    stage_host = [torch.zeros(total, dtype=torch.uint8).pin_memory() for _ in range(NBUF)]
    stage_dev = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    dev_in = [{} for _ in range(NBUF)]
    for bb in range(NBUF):
        for n, x in srcs:
            nb = x.numel() * x.element_size()
            stage_host[bb][offs[n]:offs[n] + nb].copy_(x.cpu().contiguous().view(-1).view(torch.uint8))
            dev_in[bb][n] = stage_dev[bb][offs[n]:offs[n] + nb].view(x.dtype).view(x.shape)
    outs = [out] + [torch.empty_like(out) for _ in range(NBUF - 1)]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NBUF)]
    h2d = sum(x.numel() * x.element_size() for _, x in srcs)
    d2h = out_host[0].numel() * out_host[0].element_size()
    K_e2e = max(10, K // 4)

    def e2e_serial_step():
        stage_dev[0].copy_(stage_host[0], non_blocking=True)
        enqueue(args.path, *[dev_in[0][n] for n in names])
        out_host[0].copy_(out, non_blocking=True)

    def e2e_pipelined(n_steps):
        return pipelined_steps(
            stream, n_steps,
            lambda bb: stage_dev[bb].copy_(stage_host[bb], non_blocking=True),
            lambda bb: enqueue(args.path, *[dev_in[bb][n] for n in names], o=outs[bb]),
            lambda bb: out_host[bb].copy_(outs[bb], non_blocking=True),
            hold_ms=queue_ahead_ms(4 * host_ms, n_steps), nbuf=NBUF)

    for _ in range(3):
        e2e_serial_step()
    e2e_serial_ms = timed_steps(e2e_serial_step, K_e2e, stream, 4 * host_ms) / K_e2e
    e2e_pipelined(4)
    e2e_ms = e2e_pipelined(K_e2e)
    if not torch.equal(out_host[(K_e2e - 1) % NBUF], out.cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the device output")
    del stage_host, stage_dev, dev_in, outs, out_host

    step_b = decode_b + append_b
    rec = {
        "value": round(step_b * world / (ms_step * 1e-3) / 1e9, 2), "unit": "GB/s",
        "ms_per_step": round(ms_step, 5), "steps": K,
        "dtype": "fp16" if case.q.dtype == torch.float16 else "bf16",
        "config": workload_config(case, label, world),
        "execution": {"step": "fused append+decode launch" if args.path == "fused"
                      else "kv_append then decode", "partition_size": part, "split": split,
                      "launches_per_step": launches_per_step,
                      "timed_region": "steps queued behind a bounded device-side wait before "
                                      "the start event"},
        "pct_of_peak": round(100.0 * step_b / (ms_step * 1e-3) / 1e9 / peak, 2),
        "decode_seqs_per_s": round(S * world / (ms_step * 1e-3), 1),
        "roofline": roofline,
        "e2e": {"value": round(step_b * world / (e2e_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "copies": "own streams, double-buffered: the next step's inputs in and this "
                          "step's output out while the next step computes",
                "serial_ms_per_step": round(e2e_serial_ms, 5),
                "serial_value": round(step_b * world / (e2e_serial_ms * 1e-3) / 1e9, 2)},
        "gpu_launches": K * launches_per_step,
        "clocks": clock_rec,
    }
    if extras:
        # The other path, briefly, for comparison (not the headline).
        other = "separate" if args.path == "fused" else "fused"
        n_alt = max(20, K // 10)
        for _ in range(3):
            enqueue(other, *dev_args)
        alt_ms = timed_steps(lambda: enqueue(other, *dev_args), n_alt, stream, host_ms) / n_alt
        rec["other_path"] = {"path": other, "ms_per_step": round(alt_ms, 5), "steps": n_alt}
        # Contiguous baseline: the same tokens with each sequence reserved at
        # max_context_len and no block table; the ratio of the two decode
        # times is the cost of the indirection.
        rec["contiguous_baseline"] = contiguous_baseline(pkv, case, out, part, dev, stream,
                                                         max(20, K // 10))
        rec["cache_ops"] = cache_ops_bench(pkv, case, dev, stream, peak)
        if rank == 0 and world == 1:
            rate, n, secs = oracle_sample_rate(case, k_new, v_new, slots, args.cpu_seconds)
            host = host_info()
            rec["cpu_baseline"] = {
                "value": round(rate, 4), "unit": "GB/s", "cores": host["cores"], "kind": "oracle",
                "cpu_model": host["cpu_model"], "blas": host["blas"],
                "blas_threads": host["blas_threads"],
                "sample": f"{n} whole sequences of this workload in random order (append + decode "
                          f"in fp64), {secs:.1f} s"}
    del case, k_new, v_new, slots, out, workspace
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local_rank):
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    set_decode_path(args)
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    K = args.steps
    main = decode_record(pkv, args, args.workload, dev, stream, world, K, True, rank)
    line = {"metric": METRIC, "value": main["value"], "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": main["dtype"], "data": "synthetic"}
    line.update({k: v for k, v in main.items() if k not in line and k != "steps"})
    if args.workload == "opt13b" and args.num_seqs is None:
        # The grouped-query workload is the second shape the target names; it
        # is measured the same way and reported beside the headline.
        line["gqa4k"] = decode_record(pkv, args, "gqa4k", dev, stream, world, K, False, rank)
        # The other configurations, each in its own (shorter) form, so that
        # one default run measures every one of them: the decode sweep at
        # blocks of 16 (batches 8 and 64, contexts 1k, 8k, 32k), the
        # shared-prompt serving step, and chunked prefill on the tensor cores.
        sw = sweep_line(args, rank, world, local_rank, block_sizes=(16,))
        line["sweep_b16"] = {"rows": sw["sweep"], "l2": sw["config"]["l2"],
                             "empty_kernel_ms": sw["empty_kernel_ms"], "clocks": sw["clocks"]}
        sh = shared_line(args, rank, world, local_rank)
        line["shared_prefix"] = {k: sh[k] for k in (
            "value", "unit", "ms_per_step", "steps_per_s", "steps", "device_ms_per_step",
            "kernel_ms_last_step", "logical_gbs_kernel", "dram_bytes_kernel", "dram_gbs_kernel",
            "allocator_us_per_step", "first_step", "held_kv_bytes", "logical_kv_bytes_per_step",
            "config", "clocks")}
        pf = prefill_line(args, rank, world, local_rank, with_cpu=False)
        line["prefill"] = {k: pf[k] for k in (
            "metric", "value", "unit", "ms_per_step", "config", "roofline", "e2e", "clocks")}
        line["gpu_launches_note"] = ("gpu_launches counts the headline step's timed region; "
                                     "each sub-record times its own")
    if rank == 0:
        print(json.dumps(line), flush=True)


def prefill_flops(lens, chunks, num_q_heads, head_dim):
    """Algorithmic FLOPs of causal chunked attention: every (query, key<=pos)
    pair costs a D-long dot product and a D-long axpy (2 flops per MAC)."""
    total = 0
    for n, c in zip(lens, chunks):
        first = n - c  # position of the chunk's first query
        total += (c * (first + 1) + c * (c - 1) // 2) * num_q_heads * 4 * head_dim
    return total


def run_prefill(args, rank, world, local_rank):
    line = prefill_line(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


def prefill_line(args, rank, world, local_rank, with_cpu=True):
    """The chunked-prefill record (TFLOP/s of the causal attention)."""
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    from paged_kv_cache_247_gb300 import workloads as W
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    set_decode_path(args)
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.PREFILL_CHUNKS
    case, q, qs = W.prefill_chunks(device=dev, num_seqs=args.num_seqs)
    S, Hq, D = q.shape[0] // w["chunk"], q.shape[1], q.shape[2]
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def call(qd, od):
        pkv.paged_attn_prefill(od, qd, qs, case.k_cache, case.v_cache, case.block_tables,
                               case.context_lens, case.scale, case.max_context_len, w["chunk"])

    pkv.device_status(clear=True)
    W = max(3, args.warmup)
    t_host = 0.0
    for i in range(W):
        t0 = time.perf_counter()
        call(q, out)
        if i >= W // 2:
            t_host += time.perf_counter() - t0
    torch.cuda.synchronize()
    host_ms = 1e3 * t_host / (W - W // 2)
    K = args.steps
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ms = timed_steps(lambda: call(q, out), K, stream, host_ms) / K
    clock_rec = clocks.stop()
    if pkv.device_status(clear=True):
        raise RuntimeError("device status flags during the prefill bench")
    ms = max_over_ranks(ms, world)
    lens = case.context_lens.cpu().tolist()
    flops = prefill_flops(lens, [w["chunk"]] * S, Hq, D)
    tflops = flops / (ms * 1e-3) / 1e12
    # MMA work actually issued: full 128x128 tiles up to each tile's last query
    group = Hq // case.k_cache.shape[1]
    gp = 1
    while gp < group:
        gp *= 2
    qpt = 128 // gp
    issued = 0
    for n in lens:
        for qt in range(-(-w["chunk"] // qpt)):
            last = n - w["chunk"] + min(w["chunk"], (qt + 1) * qpt) - 1
            issued += (last // 128 + 1) * 2 * 2 * 128 * 128 * D
    issued *= case.k_cache.shape[1]
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    # end to end: queries in from pinned host memory, output back, each step;
    # the copies run double-buffered on streams of their own (the serial form
    # is reported beside it)
    q_host = q.cpu().pin_memory()
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    q_dev = [torch.empty_like(q) for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    n_e2e = max(5, K // 4)

    def e2e_serial_step():
        q_dev[0].copy_(q_host, non_blocking=True)
        call(q_dev[0], out)
        out_host[0].copy_(out, non_blocking=True)
    e2e_serial_ms = timed_steps(e2e_serial_step, n_e2e, stream, 4 * host_ms) / n_e2e
    e2e_ms = pipelined_steps(stream, n_e2e,
                             lambda bb: q_dev[bb].copy_(q_host, non_blocking=True),
                             lambda bb: call(q_dev[bb], outs[bb]),
                             lambda bb: out_host[bb].copy_(outs[bb], non_blocking=True),
                             hold_ms=queue_ahead_ms(4 * host_ms, n_e2e))
    if not torch.equal(out_host[(n_e2e - 1) & 1], out.cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the device output")
    line = {
        "metric": "paged chunked-prefill attention TFLOP/s (causal, algorithmic)",
        "value": round(tflops * world, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"chunked prefill: {S} seqs x {w['chunk']} queries over ctx "
                   f"{w['ctx']}, 32q/8kv, D=128, B=16", "algorithmic_flops": flops,
                   "mma_flops_issued": issued},
        "roofline": {"kernel": "paged_prefill_kernel (tcgen05)", "bound": "tensor",
                     "achieved": round(tflops, 2), "peak": peak, "peak_kind": kind,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "frac_issued": round(issued / (ms * 1e-3) / 1e12 / peak, 4),
                     "traffic": ncu_traffic("paged_prefill_kernel", "prefill",
                                            PREFILL_SOURCES) if S == w["num_seqs"] else None},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": q_host.numel() * 2,
                "d2h_bytes_per_step": out_host[0].numel() * 2, "ms_per_step": round(e2e_ms, 5),
                "copies": "own streams, double-buffered: the next step's queries in and this "
                          "step's output out while the next step computes",
                "serial_ms_per_step": round(e2e_serial_ms, 5),
                "serial_value": round(flops / (e2e_serial_ms * 1e-3) / 1e12 * world, 2)},
        "gpu_launches": K, "clocks": clock_rec,
    }
    if with_cpu and rank == 0 and world == 1:
        import oracle
        n_q = 8
        tables = case.block_tables.cpu().numpy()
        nb = -(-lens[0] // case.block_size)
        ids = torch.from_numpy(tables[0, :nb].astype(np.int64)).to(dev)
        kc = case.k_cache.index_select(0, ids).float().cpu().numpy()
        vc = case.v_cache.index_select(0, ids).float().cpu().numpy()
        qq = q[w["chunk"] - n_q: w["chunk"]].float().cpu().numpy()
        t0 = time.perf_counter()
        oracle.paged_prefill_attention(qq, kc, vc, np.arange(nb)[None, :], [lens[0]],
                                       np.array([0, n_q]), case.scale)
        secs = time.perf_counter() - t0
        f_sample = prefill_flops([lens[0]], [n_q], Hq, D)
        line["cpu_baseline"] = {"value": round(f_sample / secs / 1e12, 6), "unit": "TFLOP/s",
                                "cores": cores_used(), "kind": "oracle",
                                "sample": f"the last {n_q} queries of one sequence, {secs:.2f} s"}
    del case, q, qs, out, q_host, out_host, q_dev, outs
    torch.cuda.empty_cache()
    return line


def run_shared(args, rank, world, local_rank):
    line = shared_line(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


def shared_line(args, rank, world, local_rank):
    """Parallel sampling with shared prompts (16 prompts x 8 samples): each
    timed step is the whole serving step - the native allocator's next slots
    and copy-on-write pairs and the block tables on the host, one staged copy
    of the step's inputs to the device, the copies (if any) and the fused
    append + decode launch, and the output read back.  Logical bytes are the
    K/V every sample attends over; held bytes are the blocks the pool holds."""
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    from paged_kv_cache_247_gb300 import workloads as W
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    set_decode_path(args)
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    w = W.SHARED_PREFIX
    H, D, B, n = w["num_kv_heads"], w["head_dim"], w["block_size"], w["samples"]
    dt = W.DTYPES[w["dtype"]]
    e = torch.tensor([], dtype=dt).element_size()
    prompts = W.shared_prefix_prompts()
    S = len(prompts) * n
    # The workload is a fixed number of decode steps (contexts grow by one
    # token a step): a few untimed steps, then the workload's steps timed.
    warm, K = max(3, min(args.warmup, 10)), min(args.steps, w["steps"])
    total_steps = warm + K
    seq_ids = np.arange(S, dtype=np.int64)
    nb = int(sum(-(-int(p) // B) for p in prompts) + S * (-(-total_steps // B) + 2))
    kc = torch.zeros((nb, H, B, D), dtype=dt, device=dev)
    vc = torch.zeros_like(kc)
    alloc = pkv.BlockAllocator(nb, B)
    for i, plen in enumerate(prompts.tolist()):
        pk, pv = W.new_tokens(1000 + i, plen, H, D, w["dtype"], device=dev)
        alloc.add_seq(i * n, plen)
        pkv.kv_append(pk, pv, kc, vc, torch.from_numpy(alloc.seq_slots(i * n, 0, plen)).to(dev))
        for j in range(1, n):
            alloc.fork(i * n, i * n + j)
    lens = prompts.repeat(n).astype(np.int64)
    max_blocks = -(-int(lens.max() + total_steps) // B)
    gen = torch.Generator(device="cpu").manual_seed(17)
    q_h = torch.randn((S, H, D), generator=gen).to(dt)
    k_h = torch.randn((S, H, D), generator=gen).to(dt)
    v_h = torch.randn((S, H, D), generator=gen).to(dt)
    # two pinned staging buffers (a step writes one while the other's copy
    # may still run), each: q, k_new, v_new, tables, lengths, 256-byte aligned
    parts = [("q", q_h.numel() * e), ("k", k_h.numel() * e), ("v", v_h.numel() * e),
             ("tables", S * max_blocks * 4), ("lens", S * 4)]
    offs, total = {}, 0
    for name, nbytes in parts:
        offs[name] = total
        total += -(-nbytes // 256) * 256
    stage_h = [torch.zeros(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    stage_d = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def views(buf, name, dtype, shape):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        return buf[offs[name]:offs[name] + nbytes].view(dtype).view(shape)

    for b in range(2):
        views(stage_h[b], "q", dt, q_h.shape).copy_(q_h)
        views(stage_h[b], "k", dt, k_h.shape).copy_(k_h)
        views(stage_h[b], "v", dt, v_h.shape).copy_(v_h)
    # the views of each staging buffer never change: build them once
    hv = [{"tables": views(stage_h[b], "tables", torch.int32, (S, max_blocks)),
           "lens": views(stage_h[b], "lens", torch.int32, (S,))} for b in range(2)]
    dv = [{"q": views(stage_d[b], "q", dt, q_h.shape), "k": views(stage_d[b], "k", dt, k_h.shape),
           "v": views(stage_d[b], "v", dt, v_h.shape),
           "tables": views(stage_d[b], "tables", torch.int32, (S, max_blocks)),
           "lens": views(stage_d[b], "lens", torch.int32, (S,))} for b in range(2)]
    out = torch.empty((S, H, D), dtype=dt, device=dev)
    out_h = torch.empty((S, H, D), dtype=dt).pin_memory()
    ws = torch.empty(max(16, pkv.decode_workspace_size(S, H, H, D, int(lens.max()) + total_steps + 1, 0)),
                     dtype=torch.uint8, device=dev)
    pairs_d = torch.empty((S, 2), dtype=torch.int64, device=dev)
    stats = {"alloc_s": 0.0, "copies": 0, "logical_bytes": 0}
    gpu_ev = []  # (start, end) of each timed step's device work

    def step(i, ev=None):
        b = i & 1
        done[b].synchronize()  # the copy that last read this staging buffer has ended
        t0 = time.perf_counter()
        _, pairs = alloc.append_slots(seq_ids)
        lens[:] += 1
        tables = alloc.block_table(seq_ids, max_blocks)
        stats["alloc_s"] += time.perf_counter() - t0
        hv[b]["tables"].copy_(torch.from_numpy(tables))
        hv[b]["lens"].copy_(torch.from_numpy(lens.astype(np.int32)))
        if ev is not None:
            ev[0].record(stream)
        stage_d[b].copy_(stage_h[b], non_blocking=True)
        done[b].record(stream)
        if len(pairs):
            pairs_d[:len(pairs)].copy_(torch.from_numpy(pairs), non_blocking=True)
        if len(pairs):
            pkv.block_copy(kc, vc, pairs_d[:len(pairs)])
            stats["copies"] += len(pairs)
        d = dv[b]
        pkv.paged_attn_decode_append(out, d["q"], d["k"], d["v"], kc, vc, d["tables"], d["lens"],
                                     D ** -0.5, int(lens.max()), workspace=ws)
        out_h.copy_(out, non_blocking=True)
        if ev is not None:
            ev[1].record(stream)
        stats["logical_bytes"] += int(lens.sum()) * 2 * H * D * e

    pkv.device_status(clear=True)
    t_cow = time.perf_counter()
    step(0)  # the first divergent token: every sample of a partly filled prompt block copies
    torch.cuda.synchronize()
    t_cow = time.perf_counter() - t_cow
    cow_pairs = stats["copies"]
    for i in range(1, warm):
        step(i)
    torch.cuda.synchronize()
    stats.update(alloc_s=0.0, copies=0, logical_bytes=0)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(warm, warm + K):
        ev = tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
        gpu_ev.append(ev)
        step(i, ev)
    torch.cuda.synchronize()
    elapsed = max_over_ranks(time.perf_counter() - t0, world)
    gpu_ms = float(np.mean([ev[0].elapsed_time(ev[1]) for ev in gpu_ev]))
    # The fused launch alone, on the last step's staged inputs (it rewrites
    # the same rows with the same values), queued behind a device-side wait:
    # inside the host-paced loop an event before the launch would also count
    # the host's time to issue it.
    b_last = (warm + K - 1) & 1

    def last_launch():
        d = dv[b_last]
        pkv.paged_attn_decode_append(out, d["q"], d["k"], d["v"], kc, vc, d["tables"], d["lens"],
                                     D ** -0.5, int(lens.max()), workspace=ws)
    krn_ms = time_alone(last_launch, None, stream, 20)
    krn_bytes = int(lens.sum()) * 2 * H * D * e
    # DRAM bytes of one fused launch from the committed ncu summary (a launch of
    # the timed steps, contexts within a few tokens of this one): shared prompt
    # blocks are read once per launch from DRAM and again from L2.
    dram = ncu_traffic("paged_decode_kernel:fused", "shared")
    clock_rec = clocks.stop()
    if pkv.device_status(clear=True) != 0:
        raise RuntimeError("device status flags during the shared-prefix bench")
    st = alloc.stats()
    held = st["used_blocks"] * B * 2 * H * D * e
    logical_gbs = stats["logical_bytes"] / elapsed / 1e9
    line = {
            "metric": "parallel-sampling serving step: logical K/V GB/s attended (whole step, "
                      "allocator on the host included)",
            "value": round(logical_gbs * world, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": warm, "ms_per_step": round(1e3 * elapsed / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
            "config": {"workload": f"{len(prompts)} prompts (U[{w['prompt_lo']},{w['prompt_hi']}]) "
                                   f"x {n} samples, {H} heads, D={D}, B={B}", "num_seqs": S,
                       "decode_steps": f"{warm} untimed, then {K} timed; every context grows "
                                       "by one token a step",
                       "timing": "host wall clock over the steps, device synchronised at both ends"},
            "steps_per_s": round(K / elapsed, 1),
            "device_ms_per_step": round(gpu_ms, 4),
            "device_ms_note": "input copy start to output copy end on the device clock, "
                              "including any wait for the host to issue the step's work",
            "logical_gbs_device": round(stats["logical_bytes"] / K / (gpu_ms * 1e-3) / 1e9, 1),
            "kernel_ms_last_step": round(krn_ms, 4),
            "logical_gbs_kernel": round(krn_bytes / (krn_ms * 1e-3) / 1e9, 1),
            "kernel_note": "the last step's fused append + decode launch timed alone (20 calls), "
                           "launch outside the event pair, L2 as the loop leaves it",
            "dram_bytes_kernel": dram,
            "dram_gbs_kernel": round(dram / (krn_ms * 1e-3) / 1e9, 1) if dram else None,
            "dram_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one fused launch "
                         "(profiles/traffic.json, null unless taken on the current source)",
            "allocator_us_per_step": round(1e6 * stats["alloc_s"] / K, 2),
            "first_step": {"cow_pairs": cow_pairs, "ms": round(1e3 * t_cow, 3)},
            "pool": {k: st[k] for k in st},
            "held_kv_bytes": held,
            "logical_kv_bytes_per_step": int(stats["logical_bytes"] / K),
            "clocks": clock_rec}
    alloc.close()
    del kc, vc, ws, out, stage_d
    torch.cuda.empty_cache()
    return line


def run_sweep(args, rank, world, local_rank):
    line = sweep_line(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


def sweep_line(args, rank, world, local_rank, block_sizes=None):
    """Decode over the block-size / batch / context grid: each call timed
    alone with CUDA events after reading 256 MiB (small cases fit in L2),
    algorithmic bytes / time against the HBM peak."""
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    from paged_kv_cache_247_gb300 import workloads as W
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    set_decode_path(args)
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peak_hbm()
    flush = torch.ones(32 << 20, dtype=torch.float64, device=dev)
    sw = W.SWEEP
    rows = []
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    only = tuple(int(x) for x in args.only.split(",")) if args.only else None
    for B in (block_sizes or sw["block_sizes"]):
        for S in sw["batches"]:
            for ctx in sw["ctxs"]:
                if only is not None and (B, S, ctx) != only:
                    continue
                case = W.sweep_decode(B, S, ctx, device=dev)
                Sq, Hq, D = case.q.shape
                Hkv = case.k_cache.shape[1]
                part = args.partition or pkv.decode_partition_size(Sq, Hq, Hkv, D,
                                                                   case.max_context_len)
                ws = torch.empty(max(16, pkv.decode_workspace_size(Sq, Hq, Hkv, D,
                                                                   case.max_context_len, part)),
                                 dtype=torch.uint8, device=dev)
                out = torch.empty_like(case.q)

                def call(kc=case.k_cache, vc=case.v_cache):
                    pkv.paged_attn_decode(out, case.q, kc, vc, case.block_tables,
                                          case.context_lens, case.scale, case.max_context_len,
                                          partition_size=part, workspace=ws)
                for _ in range(max(3, args.warmup)):
                    call()
                iters = max(5, min(args.steps, 30))
                ms = time_alone(call, flush, stream, iters)
                nbytes = step_bytes(case)[0]
                gbs = nbytes / (ms * 1e-3) / 1e9
                # Back to back, as the layers of a decode step run: calls in a
                # row over R copies of the cache (R x the K/V bytes > 3 x L2),
                # so no call finds its data in L2 and none waits behind a flush.
                reps = max(1, -(-(3 * 129 << 20) // int(nbytes)))
                copies = [(case.k_cache, case.v_cache)] + [
                    (case.k_cache.clone(), case.v_cache.clone()) for _ in range(reps - 1)]
                ctr = [0]

                def call_next():
                    kc, vc = copies[ctr[0] % reps]
                    ctr[0] += 1
                    call(kc, vc)
                for _ in range(reps + 2):
                    call_next()
                n_steady = max(3 * reps, iters)
                steady_ms = timed_steps(call_next, n_steady, stream, 0.05) / n_steady
                sgbs = nbytes / (steady_ms * 1e-3) / 1e9
                rows.append({"block_size": B, "num_seqs": S, "ctx": ctx, "partition": part,
                             "kv_bytes": int(nbytes), "ms": round(ms, 5), "GB/s": round(gbs, 1),
                             "frac": round(gbs / peak, 4), "steady_ms": round(steady_ms, 5),
                             "steady_frac": round(sgbs / peak, 4), "steady_copies": reps})
                del case, ws, out, copies
                torch.cuda.empty_cache()
    floor = launch_floor_ms(flush, stream, max(5, min(args.steps, 30)))
    clock_rec = clocks.stop()
    if pkv.device_status(clear=True) != 0:
        raise RuntimeError("device status flags during the sweep")
    ref = next((r for r in rows if r["block_size"] == 16 and r["num_seqs"] == 64
                and r["ctx"] == 8192), rows[-1])
    return {
            "metric": "paged decode attention HBM GB/s across block sizes, batches and contexts",
            "value": ref["GB/s"], "unit": "GB/s", "n_gpus": world, "steps": iters,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode sweep: 32q/8kv, D=128, bf16; value at B=16, 64 seqs, "
                                   "ctx 8192", "l2": "ms: flushed (256 MiB read) before every "
                                   "call; steady_ms: calls back to back over copies of the cache "
                                   "that together exceed 3 x L2",
                       "launch": "ms: queued behind a device-side wait, outside the timed "
                                 "region; steady_ms: back to back, as the layers of a step"},
            "roofline": {"bound": "hbm", "achieved": ref["GB/s"], "peak": peak, "unit": "GB/s",
                         "frac": ref["frac"], "peak_kind": peak_kind, "traffic": None},
            "sweep": rows, "empty_kernel_ms": round(floor, 5), "clocks": clock_rec}


def run_prefill_shapes(args, rank, world, local_rank):
    """Chunked prefill across shapes: query-head groups (MHA to 8), head sizes,
    chunk lengths (long chunks, short chunks at the end of long contexts,
    whole prompts) and dtypes.  Each case is K launches back to back; TFLOP/s
    of the causal attention's algorithmic work against the measured bf16
    tensor peak.  `--only N` runs the N-th case alone (for profiler captures)."""
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    from paged_kv_cache_247_gb300 import workloads as W
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    rng = np.random.default_rng(11)
    prompts = [int(x) for x in rng.integers(100, 701, size=16)]
    # (label, Hq, Hkv, D, B, dtype, context lengths, chunk lengths)
    cases = [
        ("GQA 32/8, D=128: 8 x 2048 queries over 4096", 32, 8, 128, 16, "bf16",
         [4096] * 8, [2048] * 8),
        ("MHA 40/40, D=128 (OPT-13B heads): 8 x 2048 over 4096", 40, 40, 128, 16, "fp16",
         [4096] * 8, [2048] * 8),
        ("group 8 (64/8), D=128: 8 x 2048 over 4096", 64, 8, 128, 16, "bf16",
         [4096] * 8, [2048] * 8),
        ("GQA 32/8, D=64: 8 x 2048 over 4096", 32, 8, 64, 16, "bf16",
         [4096] * 8, [2048] * 8),
        ("short chunks, GQA 32/8, D=128: 64 x 256 over 4096", 32, 8, 128, 16, "bf16",
         [4096] * 64, [256] * 64),
        ("long context, GQA 32/8, D=128: 2 x 8192 over 32768", 32, 8, 128, 16, "bf16",
         [32768] * 2, [8192] * 2),
        ("whole prompts, MHA 40/40, D=128: 16 prompts of 100-700 tokens", 40, 40, 128, 16,
         "fp16", prompts, prompts),
    ]
    pick = [int(args.only)] if args.only else range(len(cases))
    rows = []
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    iters = max(5, min(args.steps, 20))
    for ci in pick:
        label, hq, hkv, D, B, dt, lens, chunks = cases[ci]
        case = W.make_decode_case(700 + ci, len(lens), hq, hkv, D, B, dt, lens,
                                  pool_factor=1.0, device=dev)
        qs = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32,
                          device=dev)
        gen = torch.Generator(device=dev).manual_seed(ci)
        q = torch.randn((int(qs[-1]), hq, D), generator=gen, device=dev).to(case.q.dtype)
        out = torch.empty_like(q)
        max_chunk = max(chunks)

        def call():
            pkv.paged_attn_prefill(out, q, qs, case.k_cache, case.v_cache, case.block_tables,
                                   case.context_lens, case.scale, case.max_context_len,
                                   max_chunk)
        t_host = 0.0
        for i in range(max(3, args.warmup)):
            t0 = time.perf_counter()
            call()
            t_host += time.perf_counter() - t0
        torch.cuda.synchronize()
        host_ms = 1e3 * t_host / max(3, args.warmup)
        ms = timed_steps(call, iters, stream, host_ms) / iters
        flops = prefill_flops(lens, chunks, hq, D)
        tf = flops / (ms * 1e-3) / 1e12
        rows.append({"case": label, "dtype": dt, "algorithmic_flops": flops,
                     "ms": round(ms, 5), "TFLOP/s": round(tf, 1), "frac": round(tf / peak, 4)})
        del case, q, out
        torch.cuda.empty_cache()
    clock_rec = clocks.stop()
    if pkv.device_status(clear=True) != 0:
        raise RuntimeError("device status flags during the prefill shape sweep")
    if rank == 0:
        print(json.dumps({
            "metric": "paged chunked-prefill attention TFLOP/s across shapes (causal, algorithmic)",
            "value": rows[0]["TFLOP/s"], "unit": "TFLOP/s", "n_gpus": world, "steps": iters,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16/fp16 (per case)", "data": "synthetic",
            "config": {"workload": "chunked prefill shape sweep", "B": 16,
                       "timing": "launches back to back between two events",
                       "peak": peak, "peak_kind": kind},
            "cases": rows, "clocks": clock_rec}), flush=True)


def run_groups(args, rank, world, local_rank):
    """Decode across query-head group sizes over one KV cache shape (8 KV heads
    of 128, bf16, 4,096 tokens per sequence): each call timed alone after
    reading 256 MiB; algorithmic bytes (each K/V byte once per KV head) /
    time against the HBM peak.  `--group G` runs one size only (for profiler
    captures)."""
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import build as _build
    from paged_kv_cache_247_gb300 import workloads as W
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build_library()
    set_decode_path(args)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peak_hbm()
    flush = torch.ones(32 << 20, dtype=torch.float64, device=dev)
    S = args.num_seqs or 32
    groups = [args.group] if args.group else [1, 2, 4, 8, 16, 32]
    rows = []
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for G in groups:
        case = W.make_decode_case(6, S, 8 * G, 8, args.head_dim, args.block_size, "bf16",
                                  [4096] * S, device=dev)
        Sq, Hq, D = case.q.shape
        part = args.partition or pkv.decode_partition_size(Sq, Hq, 8, D, case.max_context_len)
        ws = torch.empty(max(16, pkv.decode_workspace_size(Sq, Hq, 8, D, case.max_context_len,
                                                           part)), dtype=torch.uint8, device=dev)
        out = torch.empty_like(case.q)

        def call():
            pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                                  case.context_lens, case.scale, case.max_context_len,
                                  partition_size=part, workspace=ws)
        for _ in range(max(3, args.warmup)):
            call()
        iters = max(5, min(args.steps, 30))
        ms = time_alone(call, flush, stream, iters)
        nbytes = step_bytes(case)[0]
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows.append({"group": G, "num_q_heads": Hq, "partition": part, "kv_bytes": int(nbytes),
                     "ms": round(ms, 5), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "kernel": "paged_decode_tc_kernel" if pkv.decode_uses_tensor_cores(
                         Sq, Hq, 8, D, case.max_context_len, part) else "paged_decode_kernel",
                     "traffic": ncu_traffic(f"paged_decode_tc_kernel:g{G}", "groups",
                                            DECODE_TC_SOURCES)})
        del case, ws, out
        torch.cuda.empty_cache()
    clock_rec = clocks.stop()
    if pkv.device_status(clear=True) != 0:
        raise RuntimeError("device status flags during the group sweep")
    if rank == 0:
        print(json.dumps({
            "metric": "paged decode attention HBM GB/s across query-head group sizes",
            "value": rows[-1]["GB/s"], "unit": "GB/s", "n_gpus": world, "steps": iters,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"decode, {S} seqs x 4096 tokens, 8 KV heads of {args.head_dim}, bf16, "
                                   f"B={args.block_size}, query heads 8 x group", "l2": "flushed (256 MiB read) "
                                   "before every call",
                       "launch": "queued behind a device-side wait, outside the timed region"},
            "groups": rows, "clocks": clock_rec}), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("gloo")
    try:
        if args.workload == "prefill":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the reference arm is timed on the decode workloads"}))
            else:
                run_prefill(args, rank, world, local_rank)
        elif args.workload == "prefill_shapes":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the reference arm is timed on the decode workloads"}))
            else:
                run_prefill_shapes(args, rank, world, local_rank)
        elif args.workload == "shared":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the reference arm is timed on the decode workloads"}))
            else:
                run_shared(args, rank, world, local_rank)
        elif args.workload == "groups":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the reference arm is timed on the decode workloads"}))
            else:
                run_groups(args, rank, world, local_rank)
        elif args.workload == "sweep":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the reference arm is timed on the decode workloads"}))
            else:
                run_sweep(args, rank, world, local_rank)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
