#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on GB300.

One step = one decode step of a continuous-batching layer on the decode-batch
workload (64 sequences, Llama-3.1-8B attention shape: 32 q / 8 kv heads,
d128, bf16, block size 16, cache lengths uniform in 1024..16384): the 64 new
tokens' K/V are written into the paged cache by slot mapping, then paged
decode attention runs over the updated cache.  The headline value is the
step's algorithmic HBM bytes per second (attended K/V + Q + O of the decode,
plus the written rows read and stored), i.e. paged-decode HBM GB/s.

Also measured in the same run (``also``): the long-context decode workload
(8 x 131072 tokens, 64 q / 8 kv heads) with bf16, FP8-E4M3 and INT8 caches,
the causal varlen prefill workload (TFLOP/s; packed, paged and paged FP8), the
mixed chunked batch, the fused append + decode step, speculative verification,
copy-on-write and a KV-write sweep.

``--impl reference`` times the CPU oracle (fp64 NumPy) on bounded samples of
the same workload, as the reference arm.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
``torch.distributed.run`` every rank runs its own replica (no collective on
the data path) and rank 0 prints one JSON line.
"""

import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s (% of peak) & tokens/s; varlen prefill TFLOP/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 7900.0       # GB300 datasheet HBM3e bandwidth (context beside the measured copy peak)
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 datasheet dense bf16 (context beside the measured cuBLAS peak)
L2_BYTES = 126 * 2 ** 20


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profile_traffic(kernel_key):
    """Per-launch DRAM bytes from a committed ncu summary, or None if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    import hashlib
    try:
        rows = {}
        with open(path) as f:
            for line in f:
                line = line.strip()
                if not line or line.startswith("#"):
                    continue
                key, src, digest, nbytes = line.split()[:4]
                rows[key] = (src, digest, float(nbytes))
        if kernel_key not in rows:
            return None
        src, digest, nbytes = rows[kernel_key]
        with open(os.path.join(ROOT, src), "rb") as f:
            now = hashlib.sha256(f.read()).hexdigest()[:16]
        return nbytes if now == digest else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        try:
            props = torch.cuda.get_device_properties(device)
            uuid = str(getattr(props, "uuid", "") or "")
            sel = ["-i", "GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid] if uuid else []
            self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms",
                        "200"] + sel
        except Exception:
            self.cmd = None

    def start(self):
        if not self.cmd:
            return
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.6)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (one replica per rank; no collective on the data path)
# ---------------------------------------------------------------------------


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks (the slowest rank's time); the value itself when not distributed."""
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(bytes_per_rank_step: int, ms_per_step_max: float, world: int) -> float:
    """Whole-job GB/s: every rank processed its own step's bytes within the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------


def decode_bytes(wl):
    """Algorithmic HBM bytes of one decode call: attended K/V + Q + O."""
    elt = 1 if wl.cache_dtype in ("fp8_e4m3", "int8") else 2
    lens = wl.lens_before + 1
    kv = int(lens.sum()) * wl.num_kv_heads * wl.head_dim * elt * 2
    qo = 2 * wl.batch * wl.num_heads * wl.head_dim * 2
    return kv + qo


def write_bytes(wl):
    """Algorithmic bytes of the KV write: new rows read (bf16) + stored (cache dtype), K and V."""
    elt = 1 if wl.cache_dtype in ("fp8_e4m3", "int8") else 2
    row = wl.num_kv_heads * wl.head_dim
    return wl.batch * row * (2 + elt) * 2


class DecodeStep:
    def __init__(self, pkv, wl):
        self.pkv, self.wl = pkv, wl
        shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        self.kc4 = wl.k_cache.view(shape4)
        self.vc4 = wl.v_cache.view(shape4)
        self.out = torch.empty_like(wl.q)
        need = pkv.lib().pkv_paged_attn_decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                                         wl.max_seqlen)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=wl.q.device)
        self.launches = 2 + (1 if need > 0 else 0)
        self.fused_launches = 1 + (1 if need > 0 else 0)
        self.before = (wl.cache_seqlens - 1).contiguous()  # tokens cached before the step

    def write(self, k_new=None, v_new=None, slots=None):
        wl = self.wl
        self.pkv.kv_cache_write(wl.k_new if k_new is None else k_new, wl.v_new if v_new is None else v_new,
                                wl.k_cache, wl.v_cache, wl.slot_mapping if slots is None else slots,
                                k_inv_scale=wl.k_inv_scale, v_inv_scale=wl.v_inv_scale)

    def fused(self, q=None, k_new=None, v_new=None, before=None, table=None, out=None):
        """The whole step in one launch: each new K/V row appended by the split-KV decode kernel itself."""
        wl = self.wl
        self.pkv.paged_attn_decode_with_kvcache(wl.q if q is None else q, wl.k_new if k_new is None else k_new,
                                                wl.v_new if v_new is None else v_new, self.kc4, self.vc4,
                                                self.before if before is None else before,
                                                wl.block_table if table is None else table, wl.scale,
                                                max_seqlen_k=wl.max_seqlen, k_scale=wl.k_scale, v_scale=wl.v_scale,
                                                k_inv_scale=wl.k_inv_scale, v_inv_scale=wl.v_inv_scale,
                                                out=self.out if out is None else out, workspace_buf=self.ws)

    def decode(self, q=None, seqlens=None, table=None, out=None):
        wl = self.wl
        self.pkv.paged_attn_decode(wl.q if q is None else q, self.kc4, self.vc4,
                                   wl.cache_seqlens if seqlens is None else seqlens,
                                   wl.block_table if table is None else table, wl.scale,
                                   max_seqlen_k=wl.max_seqlen, k_scale=wl.k_scale, v_scale=wl.v_scale,
                                   out=self.out if out is None else out, workspace_buf=self.ws)


def time_decode_steps(step, steps, warmup):
    """Device-timed loop of write+decode; returns (ms per step, mean decode-call ms)."""
    for _ in range(warmup):
        step.write()
        step.decode()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        step.write()
        ev[i][0].record()
        step.decode()
        ev[i][1].record()
    end.record()
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    dec = sum(a.elapsed_time(b) for a, b in ev) / steps
    return total / steps, dec


def time_fused_steps(step, steps, warmup):
    """Device-timed loop of the one-launch step (append + decode); returns (ms per step, mean call ms)."""
    for _ in range(warmup):
        step.fused()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        ev[i][0].record()
        step.fused()
        ev[i][1].record()
    end.record()
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    call = sum(a.elapsed_time(b) for a, b in ev) / steps
    return total / steps, call


def time_e2e(step, steps, warmup):
    """Per step: one H2D copy of the step's inputs (packed in one pinned host buffer, each tensor at a
    256-byte boundary), the one-launch step (append + decode) on device views of that buffer, and a D2H
    read of the step's output.  Both copies run on copy streams with two device buffers each: the
    next step's inputs are copied while this step's kernels run, and this step's output is read
    while the next step's run; a step's kernels wait for its own input copy.  Every copy of the
    timed steps is issued and has completed inside the timed region."""
    wl = step.wl
    names = ("q", "k_new", "v_new", "before", "block_table")
    srcs = [(step.before if name == "before" else getattr(wl, name)).contiguous() for name in names]
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dev_buf = [torch.empty(total, dtype=torch.uint8, device=wl.q.device) for _ in range(2)]
    dev = [{}, {}]
    for name, t, off in zip(names, srcs, offs):
        nb = t.numel() * t.element_size()
        host_buf[off:off + nb].copy_(t.cpu().view(-1).view(torch.uint8))
        for b in range(2):
            dev[b][name] = dev_buf[b][off:off + nb].view(t.dtype).view(t.shape)
    out_dev = [step.out, torch.empty_like(step.out)]
    out_host = [torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = total
    d2h = out_host[0].numel() * out_host[0].element_size()
    cur = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=wl.q.device)    # H2D
    down = torch.cuda.Stream(device=wl.q.device)  # D2H
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    decoded = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    count = [0]

    def copy_in(i):
        b = i & 1
        if i >= 2:
            up.wait_event(used[b])  # the kernels of two steps back have read this input buffer
        with torch.cuda.stream(up):
            dev_buf[b].copy_(host_buf, non_blocking=True)
        copied[b].record(up)

    def one(last):
        i = count[0]
        b = i & 1
        cur.wait_event(copied[b])
        if i >= 2:
            cur.wait_event(read[b])  # the read of two steps back has left this output buffer
        step.fused(dev[b]["q"], dev[b]["k_new"], dev[b]["v_new"], dev[b]["before"], dev[b]["block_table"],
                   out=out_dev[b])
        used[b].record(cur)
        decoded[b].record(cur)
        if not last:
            copy_in(i + 1)
        down.wait_event(decoded[b])
        with torch.cuda.stream(down):
            out_host[b].copy_(out_dev[b], non_blocking=True)
        read[b].record(down)
        count[0] += 1

    copy_in(count[0])
    for w in range(warmup):
        one(w == warmup - 1)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    cur.wait_event(start)
    up.wait_stream(cur)  # the first input copy starts inside the timed region
    copy_in(count[0])
    for k in range(steps):
        one(k == steps - 1)
    cur.wait_stream(down)  # every output read is inside the timed region
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def sampled_oracle_decode(wl, seqs):
    """Copy the sampled sequences' blocks to the host and run the oracle on them."""
    import oracle as O
    table = wl.block_table.cpu().numpy()
    lens = wl.cache_seqlens.cpu().numpy()
    blocks = sorted({int(x) for s in seqs for x in table[s][:-(-int(lens[s]) // wl.block_size)]})
    remap = {b: i for i, b in enumerate(blocks)}
    idx = torch.tensor(blocks, device=wl.q.device)
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)

    def host_bits(t):
        t = t.view(shape4)[idx].reshape(-1, wl.num_kv_heads, wl.head_dim).cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    kc, vc = host_bits(wl.k_cache), host_bits(wl.v_cache)
    tsub = np.full_like(table, -1)
    for s in seqs:
        n = -(-int(lens[s]) // wl.block_size)
        tsub[s, :n] = [remap[int(x)] for x in table[s][:n]]
    q = wl.q.cpu().view(torch.int16).numpy().view(np.uint16)
    return O, q, kc, vc, lens, tsub


def _oracle_worker(task):
    """One process of the all-cores oracle timing: the oracle, as it stands, on a few
    sequences of its own with the decode batch's shapes (32 q / 8 kv heads, d128,
    block size 16) and length distribution (uniform in 1024..16384), seeded; so no
    cache is copied between processes."""
    seed, budget_s, n_seqs = task
    import oracle as O
    rng = np.random.default_rng(seed)
    hq, hkv, d, bs = 32, 8, 128, 16
    lens = rng.integers(1024, 16384, size=n_seqs, endpoint=True)
    nblk = -(-lens // bs)
    perm = rng.permutation(int(nblk.sum())).astype(np.int32)
    table = np.full((n_seqs, int(nblk.max())), -1, np.int32)
    off = 0
    for i, n in enumerate(nblk):
        table[i, :n] = perm[off:off + n]
        off += n

    def bf16_bits(shape):  # N(0,1) fp32 rounded to nearest-even bf16, as bit patterns
        x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32).view(np.uint32)
        return ((x + 0x7FFF + ((x >> 16) & 1)) >> 16).astype(np.uint16).reshape(shape)

    kc = bf16_bits((int(nblk.sum()) * bs, hkv, d))
    vc = bf16_bits((int(nblk.sum()) * bs, hkv, d))
    q = bf16_bits((n_seqs, hq, d))
    done, count = 0, 0
    t0 = time.perf_counter()
    while True:
        s = count % n_seqs
        O.paged_attn_decode(q, kc, vc, lens, table, bs, d ** -0.5, "bf16", 1.0, 1.0, seqs=[s])
        done += int(lens[s]) * hkv * d * 2 * 2 + 2 * hq * d * 2
        count += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0, count


def oracle_decode_rate_all_cores(budget_s, seqs_per_worker=2):
    """Oracle throughput with one single-threaded process per host core (spawned, so no
    process is forked after the CUDA context exists): summed bytes / longest worker window."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(2003 + w, budget_s, seqs_per_worker) for w in range(n)])
    return sum(r[0] for r in res) / max(r[1] for r in res), n, sum(r[2] for r in res)


def cpu_model():
    """The host CPU's model name (x86), or its implementer and part ids (Arm cpuinfo has no name)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("cpu implementer") and fields.get("cpu part"):
        return (f"{platform.machine()} CPU implementer {fields['cpu implementer']} "
                f"part {fields['cpu part']}")
    return platform.processor() or platform.machine()


def oracle_decode_rate(wl, budget_s, max_seqs=64):
    """Oracle throughput (algorithmic bytes/s): whole sampled sequences, cycled until the budget is spent."""
    order = [int(s) for s in np.random.default_rng(0).permutation(wl.batch)[:max_seqs]]
    O, q, kc, vc, lens, tsub = sampled_oracle_decode(wl, order)
    elt = 1 if wl.cache_dtype == "fp8_e4m3" else 2
    done_bytes, done_tok, nseq = 0, 0, 0
    t0 = time.perf_counter()
    while True:
        s = order[nseq % len(order)]
        L = int(lens[s])
        O.paged_attn_decode(q, kc, vc, lens, tsub, wl.block_size, wl.scale, wl.cache_dtype, wl.k_scale,
                            wl.v_scale, seqs=[s])
        done_bytes += L * wl.num_kv_heads * wl.head_dim * elt * 2 + 2 * wl.num_heads * wl.head_dim * 2
        done_tok += L
        nseq += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done_bytes / dt, nseq, done_tok, dt


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------


def run_pkv(args, rank, world, device):
    from paged_kv_cache_200_gb300 import build as B
    from paged_kv_cache_200_gb300 import pkv
    from paged_kv_cache_200_gb300 import workloads as W

    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    if world > 1:
        torch.distributed.barrier()
    pkv.lib()
    pk = peaks()

    wl = W.decode_batch(device=device)
    step = DecodeStep(pkv, wl)
    nbytes = decode_bytes(wl) + write_bytes(wl)

    # CPU baseline (rank 0 only): the oracle on a bounded sample of the same workload
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, nseq, ntok, dt = oracle_decode_rate(wl, budget_s=args.cpu_budget)
        cpu = {"value": rate / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{nseq} whole-sequence decodes drawn from the decode batch ({ntok} cached tokens, "
                         f"all 32 heads), fp64 NumPy, single thread, {dt:.1f} s",
               "cpu_model": cpu_model()}
        if args.cpu_all_cores_budget > 0:
            try:
                rate_n, ncores, nseq_n = oracle_decode_rate_all_cores(args.cpu_all_cores_budget)
                cpu["all_cores"] = {
                    "value": rate_n / 1e9, "unit": "GB/s", "cores": ncores,
                    "sample": f"{nseq_n} whole-sequence decodes, one single-threaded oracle process per core, "
                              f"each on 2 seeded sequences of the decode batch's shapes and length distribution, "
                              f"{args.cpu_all_cores_budget:.0f} s"}
            except Exception as e:  # the single-thread figure stands alone
                cpu["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}

    clocks = ClockSampler(device)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ms, dec_ms = time_fused_steps(step, args.steps, args.warmup)
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, device)
    if world > 1:
        torch.distributed.barrier()

    e2e_ms, h2d, d2h = time_e2e(step, max(1, min(args.steps, args.e2e_steps)), 3)
    e2e_ms = max_over_ranks(e2e_ms, device)

    also, legs = {}, {}
    if not args.no_extra:
        also, legs = extra_workloads(pkv, W, device, pk, args)

    dec_bytes = decode_bytes(wl)
    achieved = nbytes / (dec_ms * 1e-3) / 1e9
    traffic = profile_traffic("paged_decode_split_append_bf16_d128")
    result = {
        "metric": METRIC,
        "value": job_throughput_gbs(nbytes, ms_max, world),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q, seeded lengths and permuted block pool)",
        "config": {
            "workload": "decode_batch64: 64 seqs, cached lengths U[1024,16384] + 1 new token each, 32 q / 8 kv "
                        "heads, head_dim 128, bf16 cache, block_size 16, permuted pool; step = KV write of the 64 "
                        "new tokens + paged decode attention, as one launch (each new row appended by the split-KV "
                        "decode kernel; the two-launch step is in also.decode_with_kvcache)",
            "batch": wl.batch,
            "attended_tokens": int((wl.lens_before + 1).sum()),
            # share of the block pool holding tokens (the pool has exactly the blocks the lengths need)
            "pool_utilisation": float((wl.lens_before + 1).sum()) / float(wl.num_blocks * wl.block_size),
            "bytes_per_step": nbytes,
            "l2": "inputs larger than L2 (%.2f GB of K/V read per step)" % (dec_bytes / 1e9),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": world * wl.batch / (ms_max * 1e-3),
        "roofline": {
            "kernel": "paged_attn_decode_with_kvcache (split-KV kernel with the step's K/V append + combine, "
                      "one call)",
            "bound": "hbm",
            "achieved": achieved,
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"],
            "traffic": traffic,
            "algorithmic_bytes": nbytes,
            "launch_ms": dec_ms,
            "peak_source": pk["source"] + " copy bandwidth (hbm_gbs)",
            "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
        },
        "e2e": {"value": job_throughput_gbs(nbytes, e2e_ms, world), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": step.fused_launches * args.steps,
        "clocks": clk,
    }
    if cpu is not None:
        result["cpu_baseline"] = cpu
    result["also"] = also
    # compact figures of the other workloads last, so that the end of the line carries them
    result["legs"] = legs
    return result


def _r(x, n=4):
    """x rounded to n significant digits (keeps the compact figures short)."""
    return float(f"{x:.{n}g}") if isinstance(x, float) else x


def extra_workloads(pkv, W, device, pk, args):
    """The other workloads: full records (``also``) and compact figures (``legs``)."""
    also, legs = {}, {}
    for dt in ("bf16", "fp8_e4m3", "int8"):
        wl = W.long_decode(device=device, cache_dtype=dt)
        step = DecodeStep(pkv, wl)
        steps = max(10, min(200, args.steps // 10))
        ms, dec_ms = time_decode_steps(step, steps, 3)
        b = decode_bytes(wl)
        ach = b / (dec_ms * 1e-3) / 1e9
        also[f"long_decode_{dt}"] = {
            "workload": "8 seqs x 131072 cached tokens (+1), 64 q / 8 kv heads, d128, block 32, " + dt + " cache",
            "decode_ms": dec_ms, "step_ms": ms, "GB_per_s": ach, "frac_of_hbm_peak": ach / pk["hbm_gbs"],
            "tokens_per_s": wl.batch / (ms * 1e-3), "steps": steps}
        legs[f"long_decode_{dt}"] = {"ms": _r(dec_ms), "GB_s": _r(ach), "frac": _r(ach / pk["hbm_gbs"])}
        del step, wl
        torch.cuda.empty_cache()
    also.update(with_kvcache_workload(pkv, W, device, pk, args))
    legs["decode_with_kvcache"] = {"ms": _r(also["decode_with_kvcache"]["step_ms"]),
                                   "frac": _r(also["decode_with_kvcache"]["frac_of_hbm_peak"])}
    also.update(copy_workload(pkv, W, device, pk, args))
    also.update(write_sweep(pkv, device, pk, args))
    mq = multi_query_workload(pkv, W, device, pk, args)["multi_query_decode"]
    also["multi_query_decode"] = mq
    legs["multi_query_decode"] = {"ms": _r(mq["ms"]), "GB_s_once": _r(mq["GB_per_s"]),
                                  "frac": _r(mq["frac_of_hbm_peak"])}
    pre = prefill_workload(pkv, W, device, pk, args)
    also.update(pre)
    for key in ("varlen_prefill_packed", "varlen_prefill_paged", "varlen_prefill_paged_direct",
                "varlen_prefill_paged_fp8", "varlen_prefill_paged_fp8_direct"):
        if key in pre:
            e = pre[key]
            legs[key] = {"ms": _r(e["ms"]), "TFLOP_s": _r(e["TFLOP_per_s"]), "frac": _r(e["frac_of_bf16_peak"])}
    legs["varlen_prefill_packed"]["roofline"] = {k: _r(v) for k, v in pre["varlen_prefill_packed"]["roofline"].items()}
    mc = pre["mixed_chunked"]
    legs["mixed_chunked"] = {"ms": _r(mc["ms"]), "roof_ms": _r(mc["roofline_ms"]), "frac": _r(mc["frac_of_roofline"])}
    try:  # last: a failed graph capture must not cost the legs above
        also.update(example_latency(pkv, W, device))
        ex = also["decode_example_latency"]
        legs["decode_example_us"] = {"eager": _r(ex["eager_us_per_step"]), "graph": _r(ex["graph_us_per_step"])}
    except Exception as e:
        also["decode_example_latency"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return also, legs


def example_latency(pkv, W, device, iters=200):
    """The docs' worked example (3 sequences, 4 q / 2 kv heads, d64): one write + decode step is
    latency-bound, so it is timed eagerly (two host calls per step) and as a replayed CUDA graph
    (launch overhead hidden); no roofline applies at this size."""
    wl = W.decode_example(device=device)
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    out = torch.empty_like(wl.q)
    need = pkv.lib().pkv_paged_attn_decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                                     wl.max_seqlen)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    # what a serving loop holds across steps: the cache views, the host bound, the buffers
    kc4, vc4, max_len = kc.view(shape4), vc.view(shape4), int(wl.max_seqlen)

    def step():
        pkv.kv_cache_write(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
        pkv.paged_attn_decode(wl.q, kc4, vc4, wl.cache_seqlens, wl.block_table, wl.scale, max_seqlen_k=max_len,
                              out=out, workspace_buf=ws)

    eager_ms = time_calls(step, iters)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph_ms = time_calls(graph.replay, iters)
    return {"decode_example_latency": {
        "workload": "docs' worked example: 3 seqs (30/32/70 cached + 1), 4 q / 2 kv heads, d64, block 32; "
                    "write + decode per step",
        "eager_us_per_step": eager_ms * 1e3, "graph_us_per_step": graph_ms * 1e3, "iters": iters}}


def with_kvcache_workload(pkv, W, device, pk, args):
    """The decode-batch step as one launch (append + decode) against write + decode (two launches)."""
    wl = W.decode_batch(device=device)
    step = DecodeStep(pkv, wl)
    before = (wl.cache_seqlens - 1).contiguous()

    def fused():
        pkv.paged_attn_decode_with_kvcache(wl.q, wl.k_new, wl.v_new, step.kc4, step.vc4, before, wl.block_table,
                                           wl.scale, max_seqlen_k=wl.max_seqlen, out=step.out,
                                           workspace_buf=step.ws)

    def separate():
        step.write()
        step.decode()

    iters = max(20, min(200, args.steps // 10))
    ms_f = time_calls(fused, iters)
    ms_s = time_calls(separate, iters)
    b = decode_bytes(wl) + write_bytes(wl)
    res = {"decode_with_kvcache": {
        "workload": "decode_batch64 step (64 seqs, U[1024,16384] cached + 1 appended, 32 q / 8 kv, d128, bs16) "
                    "as one launch: append + decode", "step_ms": ms_f, "two_launch_step_ms": ms_s,
        "GB_per_s": b / (ms_f * 1e-3) / 1e9, "frac_of_hbm_peak": b / (ms_f * 1e-3) / 1e9 / pk["hbm_gbs"],
        "tokens_per_s": wl.batch / (ms_f * 1e-3), "iters": iters}}
    del step, wl
    torch.cuda.empty_cache()
    return res


def multi_query_workload(pkv, W, device, pk, args):
    """Speculative verification: 64 sequences with 4 new tokens each over U[1024,16384] cached tokens, one varlen call."""
    rng = np.random.default_rng(1008)
    prefix = rng.integers(1024, 16384, size=64, endpoint=True)
    wl = W.make_varlen_paged(np.full(64, 4), prefix, 32, 8, 128, 16, seed=1009, device=device)
    sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = wl.k_cache.view(sh), wl.v_cache.view(sh)
    need = pkv.lib().pkv_paged_attn_varlen_workspace(wl.batch, wl.total_q, 0, wl.num_heads, wl.num_kv_heads,
                                                      wl.head_dim, wl.max_len_q, wl.max_len_k, 1, 0, wl.block_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(wl.q)
    pkv.kv_cache_write(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    iters = max(10, min(100, args.steps // 20))
    ms = time_calls(lambda: pkv.paged_attn_varlen(wl.q, kc, vc, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.max_len_q,
                                                  wl.max_len_k, block_table=wl.block_table, scale=wl.scale, out=out,
                                                  workspace_buf=ws), iters)
    row = wl.num_kv_heads * wl.head_dim * 2 * 2  # K and V bytes per position
    once = int(wl.k_lens.sum()) * row            # each sequence's K/V read once
    per_query = int(sum(int(lk) - 4 + i + 1 for lk in wl.k_lens for i in range(4))) * row  # what the rows read
    res = {"multi_query_decode": {
        "workload": "64 seqs x 4 new tokens over U[1024,16384] cached tokens, 32 q / 8 kv, d128, bs16; each "
                    "sequence's 4 x 4 (query, head) rows in one split-KV decode pass, K/V read once (one varlen "
                    "call)", "ms": ms,
        "GB_per_s": once / (ms * 1e-3) / 1e9, "frac_of_hbm_peak": once / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
        "GB_per_s_incl_L2_rereads": per_query / (ms * 1e-3) / 1e9,
        "kv_bytes_once": once, "kv_bytes_read_per_query_rows": per_query, "tokens_per_s": wl.total_q / (ms * 1e-3),
        "iters": iters}}
    del wl, kc, vc, out, ws
    torch.cuda.empty_cache()
    return res


def copy_workload(pkv, W, device, pk, args):
    """Copy-on-write of 8192 shared blocks of the decode pool (32 KB per block and cache)."""
    wl = W.decode_batch(device=device)
    sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = wl.k_cache.view(sh), wl.v_cache.view(sh)
    rng = np.random.default_rng(1006)
    n = min(8192, wl.num_blocks // 2)
    perm = rng.permutation(wl.num_blocks)
    pairs = torch.from_numpy(np.stack([perm[n:2 * n], perm[:n]], axis=1).astype(np.int32)).to(device)
    iters = max(10, min(100, args.steps // 20))
    ms = time_calls(lambda: pkv.copy_blocks(kc, vc, pairs), iters)
    moved = 2 * 2 * n * kc[0].numel() * kc.element_size()  # K and V, read and write
    gbs = moved / (ms * 1e-3) / 1e9
    res = {"copy_blocks": {
        "workload": f"{n} (src, dst) block pairs of the 64-sequence decode pool, 16-token blocks, 8 kv heads x "
                    "128 bf16 (32 KB per block and cache), K and V", "ms": ms, "bytes": moved, "GB_per_s": gbs,
        "frac_of_hbm_peak": gbs / pk["hbm_gbs"], "iters": iters}}
    del wl, kc, vc
    torch.cuda.empty_cache()
    return res


def write_sweep(pkv, device, pk, args):
    """KV write at 2^14..2^18 tokens (8 kv heads x 128), bf16 and FP8, into a permuted pool of as many slots."""
    res = {}
    iters = max(10, min(50, args.steps // 40))
    g = torch.Generator(device=device).manual_seed(1007)
    for T in (1 << 14, 1 << 16, 1 << 18):
        k = torch.randn((T, 8, 128), generator=g, device=device).to(torch.bfloat16)
        v = torch.randn((T, 8, 128), generator=g, device=device).to(torch.bfloat16)
        slots = torch.randperm(T, generator=g, device=device).to(torch.int32)
        for dt in ("bf16", "fp8_e4m3", "int8"):
            cdt = {"bf16": torch.bfloat16, "fp8_e4m3": torch.uint8, "int8": torch.int8}[dt]
            kc = torch.empty((T, 8, 128), dtype=cdt, device=device)
            vc = torch.empty_like(kc)
            ms = time_calls(lambda: pkv.kv_cache_write(k, v, kc, vc, slots, k_inv_scale=0.25, v_inv_scale=0.25),
                            iters)
            moved = 2 * T * 8 * 128 * (2 + kc.element_size())  # read bf16, write the cache type; K and V
            gbs = moved / (ms * 1e-3) / 1e9
            res[f"write_{T}_{dt}"] = {"tokens": T, "ms": ms, "GB_per_s": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"]}
            del kc, vc
        del k, v, slots
        torch.cuda.empty_cache()
    return res


def causal_pairs(q_lens, k_lens):
    """Visible (query, key) pairs under bottom-right causal alignment."""
    tot = 0
    for lq, lk in zip(q_lens, k_lens):
        lq, lk = int(lq), int(lk)
        i = np.arange(lq, dtype=np.int64)
        tot += int(np.clip(i + lk - lq + 1, 0, lk).sum())
    return tot


def time_calls(fn, iters, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def prefill_workload(pkv, W, device, pk, args):
    """The varlen prefill workload (packed and paged) and the mixed chunked-prefill batch."""
    res = {}
    iters = max(10, min(100, args.steps // 20))
    wl = W.varlen_prefill(device=device)
    flops = 4 * wl.head_dim * wl.num_heads * causal_pairs(wl.q_lens, wl.k_lens)
    out = torch.empty_like(wl.q)
    ms = time_calls(lambda: pkv.paged_attn_varlen(wl.q, wl.k, wl.v, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.max_len_q,
                                                  wl.max_len_k, scale=wl.scale, out=out), iters)
    tf = flops / (ms * 1e-3) / 1e12
    res["varlen_prefill_packed"] = {
        "workload": "8 seqs, q_len = k_len in U[128,2048] (" + ",".join(str(int(x)) for x in wl.q_lens) +
                    "), 32 q / 8 kv heads, d128, causal, packed K/V",
        "ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"], "causal_flops": flops,
        "iters": iters,
        # the call is the prep kernel (a few microseconds) and the prefill kernel, timed alone: burst peak
        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / pk["bf16_tflops"], "flops": flops, "launch_ms": ms,
                     "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS}}
    del wl, out
    wp = W.varlen_prefill(device=device, paged=True)
    shape4 = (wp.num_blocks, wp.block_size, wp.num_kv_heads, wp.head_dim)
    kc4, vc4 = wp.k_cache.view(shape4), wp.v_cache.view(shape4)
    out = torch.empty_like(wp.q)

    def paged_leg(gather, dt="bf16", wlx=wp):
        gtok = W.gather_tokens(wlx) if gather else 0
        kc, vc = wlx.k_cache.view(shape4), wlx.v_cache.view(shape4)
        ks = wlx.extra.get("k_scale", 1.0) if dt != "bf16" else 1.0
        vs = wlx.extra.get("v_scale", 1.0) if dt != "bf16" else 1.0
        kinv = wlx.extra.get("k_inv_scale", 1.0)
        vinv = wlx.extra.get("v_inv_scale", 1.0)
        need = pkv.lib().pkv_paged_attn_varlen_workspace(wlx.batch, wlx.total_q, gtok, wlx.num_heads,
                                                          wlx.num_kv_heads, wlx.head_dim, wlx.max_len_q,
                                                          wlx.max_len_k, 1, 2 if dt != "bf16" else 0,
                                                          wlx.block_size)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)

        def step():
            pkv.kv_cache_write(wlx.k_new, wlx.v_new, wlx.k_cache, wlx.v_cache, wlx.slot_mapping, k_inv_scale=kinv,
                               v_inv_scale=vinv)
            pkv.paged_attn_varlen(wlx.q, kc, vc, wlx.cu_seqlens_q, wlx.cu_seqlens_k, wlx.max_len_q, wlx.max_len_k,
                                  block_table=wlx.block_table, scale=wlx.scale, out=out, workspace_buf=ws,
                                  gather_k_tokens=gtok, k_scale=ks, v_scale=vs)

        return time_calls(step, iters)

    for key, gather, dt, what in (
            ("varlen_prefill_paged", True, "bf16", "K/V gathered into a packed buffer first (the default with a gather "
                                                   "bound)"),
            ("varlen_prefill_paged_direct", False, "bf16", "K/V read through the block table by the tile loop"),
    ):
        ms = paged_leg(gather, dt)
        tf = flops / (ms * 1e-3) / 1e12
        res[key] = {
            "workload": "same sequences written by slot mapping into a 16-token-block permuted pool, then causal "
                        "varlen attention over the paged cache, " + what + " (step = write + attention)",
            "ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"], "iters": iters}
    wf = W.to_fp8_cache(wp)
    ms = paged_leg(True, "fp8_e4m3", wf)
    tf = flops / (ms * 1e-3) / 1e12
    res["varlen_prefill_paged_fp8"] = {
        "workload": "same, FP8 E4M3 cache (per-tensor scales; write quantises, prefill widens the gathered codes)",
        "ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"], "iters": iters}
    ms = paged_leg(False, "fp8_e4m3", wf)
    tf = flops / (ms * 1e-3) / 1e12
    res["varlen_prefill_paged_fp8_direct"] = {
        "workload": "same FP8 E4M3 cache, no gather bound: the tile loop reads the one-byte pages and widens them "
                    "to f16 in shared memory (f16 MMAs)",
        "ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"], "iters": iters}
    del wp, wf, kc4, vc4, out
    torch.cuda.empty_cache()

    wm = W.mixed_chunked(device=device)
    shape4 = (wm.num_blocks, wm.block_size, wm.num_kv_heads, wm.head_dim)
    kc4, vc4 = wm.k_cache.view(shape4), wm.v_cache.view(shape4)
    gtok = W.gather_tokens(wm)
    need = pkv.lib().pkv_paged_attn_varlen_workspace(wm.batch, wm.total_q, gtok, wm.num_heads, wm.num_kv_heads,
                                                      wm.head_dim, wm.max_len_q, wm.max_len_k, 1, 0, wm.block_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(wm.q)

    def mixed_step():
        pkv.kv_cache_write(wm.k_new, wm.v_new, wm.k_cache, wm.v_cache, wm.slot_mapping)
        pkv.paged_attn_varlen(wm.q, kc4, vc4, wm.cu_seqlens_q, wm.cu_seqlens_k, wm.max_len_q, wm.max_len_k,
                              block_table=wm.block_table, scale=wm.scale, out=out, workspace_buf=ws,
                              gather_k_tokens=gtok)

    ms = time_calls(mixed_step, iters)
    pre = wm.q_lens > 1
    mflops = 4 * wm.head_dim * wm.num_heads * causal_pairs(wm.q_lens[pre], wm.k_lens[pre])
    dec_bytes = int(wm.k_lens[~pre].sum()) * wm.num_kv_heads * wm.head_dim * 2 * 2
    t_roof = max(mflops / (pk["bf16_tflops"] * 1e12), dec_bytes / (pk["hbm_gbs"] * 1e9))
    res["mixed_chunked"] = {
        "workload": "4 x 512-query chunks over 0/2K/4K/8K prefixes (2K prefix shares the 4K chunk's blocks) + 60 "
                    "decode rows of 513..8193 keys, one varlen call after the write (chunks' K/V gathered); "
                    "32 q / 8 kv, d128, bs16",
        "ms": ms, "prefill_flops": mflops, "decode_kv_bytes": dec_bytes, "roofline_ms": t_roof * 1e3,
        "frac_of_roofline": t_roof * 1e3 / ms, "tokens_per_s": wm.total_q / (ms * 1e-3), "iters": iters}
    return res


def run_reference(args):
    """The CPU oracle on bounded samples of the decode-batch workload (rank 0 only)."""
    from paged_kv_cache_200_gb300 import workloads as W
    device = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.decode_batch(device=device)
    budget = 150.0
    # calibrate: oracle time for a 1024-token sample
    O, q, kc, vc, lens, tsub = sampled_oracle_decode(wl, list(range(wl.batch)))
    order = list(np.random.default_rng(0).permutation(wl.batch))
    t0 = time.perf_counter()
    l2 = lens.copy()
    l2[order[0]] = 1024
    O.paged_attn_decode(q, kc, vc, l2, tsub, wl.block_size, wl.scale, seqs=[order[0]])
    t1024 = time.perf_counter() - t0
    per_step = budget / (args.steps + args.warmup)
    n = int(max(16, min(int(lens.max()), 1024 * per_step / max(t1024, 1e-6))))
    elt = 2

    def one(i):
        s = order[i % len(order)]
        L = min(int(lens[s]), n)
        l3 = lens.copy()
        l3[s] = L
        O.paged_attn_decode(q, kc, vc, l3, tsub, wl.block_size, wl.scale, seqs=[s])
        return L * wl.num_kv_heads * wl.head_dim * elt * 2 + 2 * wl.num_heads * wl.head_dim * 2

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += one(args.warmup + i)
    dt = time.perf_counter() - t0
    val = nbytes / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_batch64 (same as the main arm), bounded samples: one sequence per step "
                               f"truncated to {n} cached tokens, all 32 heads"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"one sequence per step, up to {n} cached tokens, fp64 NumPy, single thread"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def ncu_case(args):
    """A small case for ncu captures: a few write+decode steps, no timing, no JSON."""
    from paged_kv_cache_200_gb300 import build as B
    from paged_kv_cache_200_gb300 import pkv
    from paged_kv_cache_200_gb300 import workloads as W
    B.build()
    if args.ncu_case == "prefill":
        # the varlen prefill workload itself (8 seqs of 128..2048 tokens, packed): ~0.2 GB of inputs
        wl = W.varlen_prefill(device="cuda")
        for _ in range(4):
            pkv.paged_attn_varlen(wl.q, wl.k, wl.v, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.max_len_q, wl.max_len_k,
                                  scale=wl.scale)
        torch.cuda.synchronize()
        log("ncu case done: prefill")
        return
    if args.ncu_case == "prefill_fp8_direct":
        # the paged prefill workload with an FP8 cache and no gather bound: the tile loop widens the pages
        wl = W.to_fp8_cache(W.varlen_prefill(device="cuda", paged=True))
        sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        pkv.kv_cache_write(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping,
                           k_inv_scale=wl.extra["k_inv_scale"], v_inv_scale=wl.extra["v_inv_scale"])
        for _ in range(4):
            pkv.paged_attn_varlen(wl.q, wl.k_cache.view(sh), wl.v_cache.view(sh), wl.cu_seqlens_q,
                                  wl.cu_seqlens_k, wl.max_len_q, wl.max_len_k, block_table=wl.block_table,
                                  scale=wl.scale, k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
        torch.cuda.synchronize()
        log("ncu case done: prefill_fp8_direct")
        return
    if args.ncu_case == "multi_query":
        # the speculative-verification workload itself (64 seqs x 4 new tokens, 1K..16K cached): 2.2 GB of K/V
        rng = np.random.default_rng(1008)
        prefix = rng.integers(1024, 16384, size=64, endpoint=True)
        wl = W.make_varlen_paged(np.full(64, 4), prefix, 32, 8, 128, 16, seed=1009, device="cuda")
        sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        pkv.kv_cache_write(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
        for _ in range(5):
            pkv.paged_attn_varlen(wl.q, wl.k_cache.view(sh), wl.v_cache.view(sh), wl.cu_seqlens_q,
                                  wl.cu_seqlens_k, wl.max_len_q, wl.max_len_k, block_table=wl.block_table,
                                  scale=wl.scale)
        torch.cuda.synchronize()
        log("ncu case done: multi_query")
        return
    if args.ncu_case == "mixed":
        # the mixed chunked batch itself (4 chunks over 0..8K prefixes + 60 decode rows, one varlen
        # call after the write, chunks gathered): about 2.5 GB of K/V pool; launch lists only
        wm = W.mixed_chunked(device="cuda")
        sh = (wm.num_blocks, wm.block_size, wm.num_kv_heads, wm.head_dim)
        gtok = W.gather_tokens(wm)
        for _ in range(4):
            pkv.kv_cache_write(wm.k_new, wm.v_new, wm.k_cache, wm.v_cache, wm.slot_mapping)
            pkv.paged_attn_varlen(wm.q, wm.k_cache.view(sh), wm.v_cache.view(sh), wm.cu_seqlens_q,
                                  wm.cu_seqlens_k, wm.max_len_q, wm.max_len_k, block_table=wm.block_table,
                                  scale=wm.scale, gather_k_tokens=gtok)
        torch.cuda.synchronize()
        log("ncu case done: mixed")
        return
    rng = np.random.default_rng(77)
    dt = {"decode_fp8": "fp8_e4m3", "decode_int8": "int8"}.get(args.ncu_case, "bf16")
    # 64 sequences of 1K..4K cached tokens: ~0.65 GB of bf16 K/V, larger than L2
    wl = W.make_decode(rng.integers(1024, 4096, 64, endpoint=True), 32, 8, 128, 16, seed=77, device="cuda",
                       cache_dtype=dt)
    step = DecodeStep(pkv, wl)
    for _ in range(4):
        step.write()
        step.decode()
    torch.cuda.synchronize()
    log("ncu case done:", args.ncu_case, "decode bytes", decode_bytes(wl))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--cpu-all-cores-budget", type=float, default=8.0,
                    help="seconds of the all-cores oracle timing (0: skip)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", choices=["decode", "decode_fp8", "decode_int8", "prefill", "multi_query",
                                           "prefill_fp8_direct", "mixed"],
                    default=None,
                    help="run a small case for an ncu capture and exit")
    args = ap.parse_args()
    if args.ncu_case:
        ncu_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    res = run_pkv(args, rank, world, device)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
