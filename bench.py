"""Benchmark of one paged decode step on GB300.

A step is one pass of the hot path over one batch: copy-on-write block copies
(when the step has any), KV append of every sequence's new token, and paged
decode attention over every cached token, new one included.

Default workload: long context (8 sequences, context lengths U[32768, 131072],
block_size 16, 32 query / 8 KV heads, head_dim 128, bf16, pool 1.1x demand,
scattered block tables; about 2.7 GB of keys and values per step, the largest
of the single-GPU workloads).  Other workloads: --workload
{decode,prefix,mixed,prefill,tiny}.

value      = unique KV bytes the decode reads per step / device step time (GB/s),
             inputs resident in HBM, L2 flushed between steps (a 256 MiB write, then a
             read pass long enough that L2 holds only clean lines).
e2e        = the same bytes / step time through the public API with host
             buffers: pinned host->device copies of the step's inputs, the
             library calls, device->host copy of the output.  The host block
             manager's bookkeeping for the step (slot reservation, tables,
             sharing groups) runs before the timed region; its own host time
             is reported beside the line as host_bookkeeping_ms.
graph_ms_per_step = the same step captured once into a CUDA graph and
             replayed (L2 flushed between replays, outside the graph).
roofline   = the decode kernel alone: algorithmic bytes per launch / its
             CUDA-event time, against the measured HBM copy bandwidth.
cpu_baseline = the float64 oracle on the host cores on a bounded sample.

--impl reference times the oracle (the only other implementation there is)
on the same workload, a bounded sample of sequences per step.
N > 1 (torchrun): every rank runs its own replica (decode needs no exchange);
value sums all ranks' bytes over the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import re
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode KV GB/s (% of GB300 HBM peak) and decode tokens/s per step"
L2_FLUSH_BYTES = 256 << 20


def _peaks(key="hbm_gbs"):
    """A measured peak (HBM GB/s, or bf16 dense TFLOP/s as a burst) and its kind."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}[key], "fallback"


def _prefill_flops(wl, lens):
    """Algorithmic FLOPs of one prefill launch: every chunk query row (token,
    query head) takes 2 D FLOPs per visible key for Q K^T and 2 D for P V; the
    query at position p sees p + 1 keys."""
    total = 0
    for L, n in zip(lens, wl.chunk_lens):
        L, n = int(L), int(n)
        total += n * (L - n) + n * (n + 1) // 2          # sum over the chunk of (position + 1)
    return 4 * wl.head_dim * wl.num_q_heads * total


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(dist, values, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the job's
    time); the values unchanged when there is no process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world, units_per_rank, ms):
    """Whole-job rate: the units every rank processed in the slowest rank's time
    (weak scaling: each rank holds its own replica of the workload)."""
    return world * units_per_rank / (ms * 1e-3)


def _workload_desc(wl):
    return (f"{wl.name}: {wl.description}; block_size {wl.block_size}, {wl.num_q_heads} q / "
            f"{wl.num_kv_heads} KV heads, head_dim {wl.head_dim}, {wl.dtype}, "
            f"{wl.num_blocks} physical blocks")


def _kv_bytes(wl, lens, groups=None):
    """Unique key+value bytes the decode reads: every cached token of every
    sequence, K and V, all KV heads, with a shared span counted once for its
    whole group when the step reads it once (pa_decode_shared)."""
    per_tok = wl.num_kv_heads * wl.head_dim * 2 * wl.elem_bytes
    tokens = int(sum(int(x) for x in lens))
    if groups is not None:
        offs, seqs, nsh = groups
        for g in range(len(nsh)):
            tokens -= (int(offs[g + 1]) - int(offs[g]) - 1) * int(nsh[g]) * wl.block_size
    return tokens * per_tok


def _algo_bytes(wl, lens):
    """Everything the decode kernel must move: KV + q + out + tables + lens."""
    S = wl.num_seqs
    q = S * wl.num_q_heads * wl.head_dim * (4 if wl.input_dtype == "f32" else 2)
    out = S * wl.num_q_heads * wl.head_dim * 4
    blocks = sum(-(-int(x) // wl.block_size) for x in lens)
    return _kv_bytes(wl, lens) + q + out + blocks * 4 + S * 4


# committed ncu summary of each workload's attention call (profiles/<name>.md)
TRAFFIC_PROFILES = {
    ("decode", "bf16"): "decode_kernel_decode_batch.md",
    ("decode", "fp8"): "decode_kernel_decode_batch_fp8.md",
    ("long", "bf16"): "decode_kernel_long_context.md",
    ("long", "fp8"): "decode_kernel_long_context_fp8.md",
    ("mixed", "bf16"): "decode_kernel_mixed.md",
    ("mixed", "fp8"): "decode_kernel_mixed_fp8.md",
    ("prefix", "bf16"): "decode_call_prefix.md",
    ("prefill", "bf16"): "prefill_tc_prefill_batch.md",
    ("prefill", "fp8"): "prefill_tc_prefill_batch_fp8.md",
    ("prefix", "fp8"): "decode_call_prefix_fp8.md",
}


def source_digest(names):
    """sha256[:16] over the named csrc files, concatenated in the given order."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_253_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_from_profile(wl):
    """DRAM bytes (read + write) per attention call from the committed ncu
    summary of this workload and pool type (captured at full size, or scaled
    from a smaller capture as the summary states); valid only while the kernel
    sources it names are unchanged (else None)."""
    name = TRAFFIC_PROFILES.get((wl.name, wl.dtype))
    if name is None:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        m_src = re.search(r"sources:\s*`([^`]+)`", text)
        srcs = m_src.group(1).split() if m_src else ["pa_decode.cu"]
        m_hash = re.search(r"source sha256\[:16\]:\s*`?([0-9a-f]{16})", text)
        m_tr = re.search(r"dram bytes per launch:\s*\|?\s*`?([0-9]+)", text)
        if m_hash and m_tr and m_hash.group(1) == source_digest(srcs):
            return int(m_tr.group(1))
    except OSError:
        pass
    return None


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        # sample file: PA_CLOCKS_DIR if set (to keep the raw samples), else the temp dir
        self.path = os.path.join(os.environ.get("PA_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"pa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except OSError:
            pass
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def _oracle_sample(wl, values, target_s=12.0, threads=None, st=None):
    """Time the oracle (step appends + float64 decode) on a bounded sample of
    sequences; returns (GB/s of KV processed, tokens/s, threads, description)."""
    import numpy as np
    from oracle import replay as orp
    from oracle.attention import default_threads
    threads = threads or default_threads()
    if st is None:
        st = orp.replay(wl, values)
    lens = st.context_lens
    order = np.random.default_rng(wl.seed).permutation(wl.num_seqs)
    # grow the sample until it takes about target_s (cycling over the batch)
    n, spent, done_tok, done_seq, done_q, calls = 1, 0.0, 0, 0, 0, 0
    pos = 0
    while spent < target_s:
        if pos >= len(order):
            pos = 0
        pick = order[pos:pos + n]
        t0 = time.perf_counter()
        if wl.chunk_lens is not None:
            orp.prefill_attention(wl, values, st, seqs=pick, threads=threads)
        else:
            orp.attention(wl, values, st, seqs=pick, threads=threads)
        dt = time.perf_counter() - t0
        spent += dt
        done_tok += int(lens[pick].sum())
        done_seq += len(pick)
        # query tokens served: one per decode, a whole chunk per prefill
        done_q += int(wl.chunk_lens[pick].sum()) if wl.chunk_lens is not None else len(pick)
        pos += len(pick)
        calls += 1
        n = max(1, min(len(order), int(n * 2)))
    per_tok = wl.num_kv_heads * wl.head_dim * 2 * wl.elem_bytes
    gbs = done_tok * per_tok / spent / 1e9
    kind = "chunk prefills" if wl.chunk_lens is not None else "decodes"
    desc = (f"{done_seq} sequence {kind} ({done_tok} cached tokens) drawn from the same "
            f"{wl.num_seqs}-sequence batch, float64 oracle, {threads} threads, {spent:.1f} s")
    return gbs, done_q / spent, threads, desc


def _parity_sample(wl, values, st, out, n=3):
    """Max-abs difference between the bench's last output and the float64
    oracle on a few sequences of the batch (the same seeded pick as the CPU
    baseline's sample), against the parity tests' tolerance."""
    import numpy as np
    from oracle import replay as orp
    from oracle.attention import default_threads
    pick = np.sort(np.random.default_rng(wl.seed).permutation(wl.num_seqs)[:n])
    got = out.double().cpu().numpy()
    if wl.chunk_lens is not None:
        cu = np.concatenate([[0], np.cumsum(wl.chunk_lens)])
        got = got[np.concatenate([np.arange(cu[s], cu[s + 1]) for s in pick])]
        ref = orp.prefill_attention(wl, values, st, seqs=pick, threads=default_threads())
    else:
        got = got[pick]
        ref = orp.attention(wl, values, st, seqs=pick, threads=default_threads())
    tol = {"f32": 1e-5, "bf16": 5e-3, "fp8": 5e-5}[wl.dtype]
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    return {"seqs": [int(s) for s in pick], "max_abs_err": err, "tol": tol, "ok": err <= tol}


def _dtype_kw(args):
    kw = {"dtype": args.kv_dtype} if args.kv_dtype else {}
    if args.num_seqs:
        kw["num_seqs"] = args.num_seqs
    return kw


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return 0
    from paged_kv_cache_253_gb300 import workloads as wls
    wl = wls.make_workload(args.workload, **_dtype_kw(args))
    values = wls.generate_values(wl, "cpu")
    per_step = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sample(wl, values, target_s=per_step / 4)
    vals, toks, descs = [], [], []
    for _ in range(args.steps):
        gbs, tps, threads, desc = _oracle_sample(wl, values, target_s=per_step)
        vals.append(gbs)
        toks.append(tps)
        descs.append(desc)
    v = sum(vals) / len(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(wl)},
        "tokens_per_s": round(sum(toks) / len(toks), 3),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": descs[-1]},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch
    from paged_kv_cache_253_gb300 import api, runtime
    from paged_kv_cache_253_gb300 import workloads as wls

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    wl = wls.make_workload(args.workload, **_dtype_kw(args))
    values = wls.generate_values(wl, f"cuda:{local}", seed=wl.seed + 1000 * rank)
    pool, bm, _ = runtime.replay_setup(wl, values, f"cuda:{local}")
    prefill = wl.chunk_lens is not None
    step = runtime.prepare_prefill(wl, values, pool, bm) if prefill else \
        runtime.prepare_step(wl, values, pool, bm)
    host_ms = step.host_ms
    lens = step.context_lens.cpu().numpy()
    # unique bytes: a shared span counts once per group whichever decode path runs
    all_groups = bm.prefix_groups(wl.batch)
    kv_bytes = _kv_bytes(wl, lens, all_groups)
    logical_kv_bytes = _kv_bytes(wl, lens)
    algo_bytes = _algo_bytes(wl, lens) - logical_kv_bytes + kv_bytes
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=f"cuda:{local}")
    flush_rd = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=f"cuda:{local}")

    def flush_l2(i):
        # write a buffer larger than L2, then read another one: the timed step
        # starts with none of its inputs in L2 and no dirty lines of the flush
        # left to write back.  The read is a uint8 sum, which torch widens
        # through a 2 GiB int64 temporary that it then reads again: long enough
        # to drain every write-back (a bare 256 MiB read left some of the
        # fill's dirty lines to the timed step, and its times scattered).
        flush.fill_(i & 0xFF)
        flush_rd.sum()

    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    if pool.get_error():
        raise RuntimeError("device error during warm-up")

    def timed(body, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n):
            flush_l2(i)                                 # evict L2 between steps
            evs[i][0].record(stream)
            body()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def decode_only():
        if prefill:
            step.attend()
        else:
            step.decode()

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = api.launch_count()
    with Clocks(local) as clk:
        step_ms = timed(step.run, args.steps)
    launches = api.launch_count() - launches0
    dec_ms = timed(decode_only, args.steps)             # the decode call alone, for the roofline
    if dist:
        dist.barrier()
    ms = sum(step_ms) / len(step_ms)
    dms = sum(dec_ms) / len(dec_ms)
    ms, dms = max_over_ranks(dist, [ms, dms], f"cuda:{local}")
    if pool.get_error():
        raise RuntimeError("device error during the timed steps")

    # ---- end to end: host buffers, pinned, through the public API ----
    # The step's inputs live in one pinned host buffer (256-byte-aligned views)
    # and go up in one copy; the result comes back in one copy.
    names = ("q", "new_k", "new_v", "slots", "pairs", "block_tables", "context_lens") + \
        (("cu_seqlens_q",) if prefill else ())
    src = {k: getattr(step, k).cpu() for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (src[k].numel() * src[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=f"cuda:{local}")

    def view(buf, k):
        t = src[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)

    for k in names:
        view(host_buf, k).copy_(src[k])
    dev = {k: view(dev_buf, k) for k in names}
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = total
    d2h = out_host.numel() * out_host.element_size()
    import dataclasses
    dstep = dataclasses.replace(step, **dev)            # the same step on the uploaded inputs
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2(i)
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_buf.copy_(host_buf, non_blocking=True)
        dstep.run()
        out_host.copy_(step.out, non_blocking=True)
        c.record(stream)
        c.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(c))
    ems = sum(e2e_ms) / len(e2e_ms)
    (ems,) = max_over_ranks(dist, [ems], f"cuda:{local}")

    # ---- the same step replayed from a CUDA graph ----
    gms = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step.run()                                  # warm: workspace sized, descriptors uploaded
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step.run()
        torch.cuda.synchronize()
        for _ in range(max(3, args.warmup)):
            graph.replay()
        gms = sum(timed(graph.replay, args.steps)) / args.steps
        (gms,) = max_over_ranks(dist, [gms], f"cuda:{local}")
        if pool.get_error():
            raise RuntimeError("device error during the graph replays")
    except RuntimeError as e:
        if "device error" in str(e):
            raise
        gms = None

    peak, peak_kind = _peaks()
    achieved = algo_bytes / (dms * 1e-3) / 1e9
    if prefill:
        flops = _prefill_flops(wl, lens)
        tpeak, tpeak_kind = _peaks("bf16_tflops")
        tflops = flops / (dms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak,
                    "peak_kind": tpeak_kind + " bf16 dense burst", "unit": "TFLOP/s",
                    "frac": round(tflops / tpeak, 4), "traffic": _traffic_from_profile(wl),
                    "kernel": "prefill (pa_prefill)", "algorithmic_flops_per_launch": flops}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                    "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": _traffic_from_profile(wl), "kernel": "decode (pa_decode)",
                    "algorithmic_bytes_per_launch": algo_bytes}
    value = job_throughput(world, kv_bytes, ms) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": _workload_desc(wl),
                   "l2": "flushed between steps (256 MiB write, then a 256 MiB uint8 sum that reads a 2 GiB int64 widening; outside the timed events)",
                   "kv_bytes_per_step": kv_bytes, "logical_kv_bytes_per_step": logical_kv_bytes,
                   "shared_groups": int(len(all_groups[2])),
                   "shared_path": bool(step.sharing()),
                   "copy_pairs_per_step": step.num_pairs,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_frac_of_" + peak_kind: round(value / world / peak, 4),
        "tokens_per_s": round(job_throughput(world, wl.num_step_tokens, ms), 1),
        "decode_ms": round(dms, 5),
        "launches_per_step": round(launches / args.steps, 2),
        "roofline": roofline,
        "e2e": {"value": round(job_throughput(world, kv_bytes, ems) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(ems, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "host block-manager bookkeeping (slots, tables, sharing groups) runs "
                        "before the timed region; its host time is host_bookkeeping_ms"},
        "host_bookkeeping_ms": round(host_ms, 4),
        "graph_ms_per_step": None if gms is None else round(gms, 5),
        "graph_value": None if gms is None else round(job_throughput(world, kv_bytes, gms) / 1e9, 2),
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import replay as orp
        cvals = {k: v.cpu() for k, v in values.items()}
        st = orp.replay(wl, cvals)
        gbs, tps, threads, desc = _oracle_sample(wl, cvals, target_s=args.cpu_seconds, st=st)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc}
        line["parity_sample"] = _parity_sample(wl, cvals, st, step.out)
        if wl.name in ("tiny", "decode"):
            # the same oracle on one host thread
            gbs1, _, _, desc1 = _oracle_sample(wl, cvals, target_s=args.cpu_seconds / 2,
                                               threads=1, st=st)
            line["cpu_baseline_1thread"] = {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                            "kind": "oracle", "sample": desc1}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long",
                    choices=["tiny", "decode", "prefix", "long", "mixed", "prefill"])
    ap.add_argument("--kv-dtype", default=None, choices=["f32", "bf16", "fp8"],
                    help="pool element type (default: the workload's own; fp8 = e4m3 codes)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the workload to this many sequences (reduced cases for "
                         "profiler captures; the bench lines use the full workloads)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=40.0,
                    help="--impl reference: total oracle seconds over warm-up and timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.workload == "prefill" and args.kv_dtype == "f32":
        ap.error("the prefill workload runs on bf16 and fp8 pools")
    if args.impl == "reference":
        return run_reference(args)
    from paged_kv_cache_253_gb300 import build
    build.build()
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
