"""KVarN decode-step benchmark on GB300.

One step = one pass of the whole hot path for every sequence of the batch: append the
new token's K/V, seal the group it completes (Hadamard rotation, 16 Sinkhorn
iterations, rounding, packing), rotate the query, attend over sink + sealed records +
tail, merge the split partials and rotate the output back -- one kvarn_decode_step
call (one kernel launch).

Workload (default): Llama-3.1-8B attention shape -- 32 query heads, 8 KV heads,
head_dim 128 -- batch 16, context 32768 + U{0..127} tail tokens per sequence, 2-bit K
and V. Synthetic data (seeded), generated on the device.

Beside it, the line carries:
- the bulk-seal rate and its FP32 roofline (`seal_roofline`), and the share of step time
  the staggered fused seals take (`seal_share`, from a back-to-back run in which every
  sequence seals several times);
- the other decode workloads (`workloads`): Qwen3-4B attention shape at 4k for its 256
  steps, the 64k long-reasoning shape at K4/V2 and K4/V4 for its 2048 steps, and the
  ragged Phi-4-14B shape (batch 64, 1k-16k, norm spikes) at 2, 4 and 8 bits, each
  through the same decode-step loop;
- a prompt-prefill leg: Qwen3-4B attention shape (32 query heads, 8 KV heads), one
  4096-token prompt through kvarn_prefill (bulk append sealing 31 groups per KV head and
  side, then causal attention of all 4096 queries over the cache), with the tensor
  roofline of the attention kernel;
- the oracle on the host cores (`cpu_baseline`, all cores and one thread).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --prefill-only

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica of the
workload on its GPU (weak scaling; the path has no exchange step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KVarN decode-attn tokens/s, achieved HBM GB/s (% roofline); seal groups/s"
WORKLOAD = "llama31_8b_gqa32x8_b16_ctx32k_k2v2"
HQ, HKV, BATCH, KB, VB, SEED = 32, 8, 16, 2, 2, 2
FLOOR = 0  # tail floor in groups (--tail-floor; 0 = the published design)


def c3_lengths():
    from quantized_kv_cache_seal_gb300 import workloads
    return list(workloads.workloads()["c3_llama31_8b_32k"].context)


def rec_bytes(b):
    return 528 + 2048 * b


def sealed_groups(n):
    """Body groups sealed at length n: group g seals when group g + FLOOR fills."""
    return max(max(n - 128, 0) // 128 - FLOOR, 0)


def step_bytes(lengths, hq=None, hkv=None, kb=None, vb=None):
    """Algorithmic HBM bytes of one decode step at the given lengths (before the step):
    sealed records read + exact fp16 K/V read + q read + out written + new token written,
    plus, for a sequence whose step seals a group, that group's tail tokens read (127
    and the new token, or all 128 with a tail floor) and the new records written and
    read. Head counts and widths default to the headline workload's."""
    hq, hkv = hq or HQ, hkv or HKV
    pair = rec_bytes(kb or KB) + rec_bytes(vb or VB)
    total = 0
    for n in lengths:
        n1 = n + 1
        sealing = sealed_groups(n1) > sealed_groups(n)
        groups = sealed_groups(n1) - (1 if sealing else 0)
        n_sink = min(n1, 128)
        n_tail = max(n1 - 128, 0) - 128 * sealed_groups(n1)
        total += hkv * (groups * pair + (n_sink + n_tail) * 512)
        total += hq * 256 * 2 + hkv * 512
        if sealing:
            total += hkv * ((127 if FLOOR == 0 else 128) * 512 + 2 * pair)
    return total


def sealing_count(lengths):
    return sum(1 for n in lengths if sealed_groups(n + 1) > sealed_groups(n))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                mx = float(parts[1])
                if t0 - 0.05 <= ts <= t1 + 0.05:
                    sm.append(float(parts[0]))
                    for name, val in zip(names, parts[4:8]):
                        if val.lower().startswith("active"):
                            reasons.add(name)
            except ValueError:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic(alg_bytes, record="decode_kernel_llama31_8b_b16_ctx32k_k2v2_traffic.json"):
    """DRAM bytes per launch from the committed ncu capture of this kernel build, scaled
    to this launch's algorithmic bytes when the record has them (the decode capture ran
    the same workload a few steps earlier; the prefill capture ran this very launch);
    None if the kernel sources changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", record)) as fh:
            rec = json.load(fh)
        h = hashlib.sha256()
        for f in rec["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        if "alg_bytes_per_launch" not in rec:
            return float(rec["dram_bytes_per_launch"])
        return float(rec["dram_bytes_per_launch"]) * alg_bytes / float(rec["alg_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def max_over_ranks(ms, pg=None, device=None):
    """The slowest rank's time for the timed region (every rank gets it); the identity
    on one rank. pg: torch.distributed (initialised) or None."""
    if pg is None:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units all ranks processed (each rank a replica of the workload: weak scaling)
    per second of the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def build_cache(torch, device, extra):
    from quantized_kv_cache_seal_gb300 import workloads
    from quantized_kv_cache_seal_gb300.cache import KVarNCache

    lengths = c3_lengths()
    cache = KVarNCache(num_layers=1, max_seqs=BATCH, num_q_heads=HQ, num_kv_heads=HKV, k_bits=KB, v_bits=VB,
                       tail_floor=FLOOR,
                       max_seq_len=max(lengths) + extra, device=device)
    ids = list(range(BATCH))
    chunk = 4096
    done = [0] * BATCH
    while any(d < n for d, n in zip(done, lengths)):
        ks, vs, counts = [], [], []
        for i, n in enumerate(lengths):
            c = min(chunk, n - done[i])
            counts.append(c)
            if c > 0:
                k, v = workloads.torch_tokens(SEED, i, done[i], c, HKV, device=device)
                ks.append(k)
                vs.append(v)
        cache.append(0, ids, counts, torch.cat(ks), torch.cat(vs))
        done = [d + c for d, c in zip(done, counts)]
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return cache, ids, lengths


def measured_tensor_peak():
    """Dense bf16 burst TFLOP/s from MEASURED_PEAKS.json (f16 mma has the same nominal
    rate), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            v = float(json.load(fh)["bf16_tflops"])
        return v, "measured bf16 dense (burst), MEASURED_PEAKS.json"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback bf16 dense"


def snapshot_leg(cache):
    """Save the headline cache to a pinned host image and restore it (into the same cache,
    which leaves its state as it was): bytes and host-clock times of both directions."""
    import torch

    from quantized_kv_cache_seal_gb300 import kvarn as K

    n = K.kvarn_snapshot_bytes(cache.handle)
    buf = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    torch.cuda.synchronize()
    saves, loads = [], []
    for _ in range(3):
        t0 = time.perf_counter()
        K.kvarn_snapshot_save(cache.handle, buf, n)
        t1 = time.perf_counter()
        K.kvarn_snapshot_load(cache.handle, buf, n)
        t2 = time.perf_counter()
        saves.append(t1 - t0)
        loads.append(t2 - t1)
    s, l = min(saves), min(loads)
    return {"bytes": n, "save_ms": s * 1e3, "load_ms": l * 1e3, "save_gbs": n / s / 1e9, "load_gbs": n / l / 1e9,
            "host_buffer": "pinned", "note": "records of every sealed group, exact regions, bookkeeping"}


PF_HQ, PF_HKV, PF_N = 32, 8, 4096  # prefill leg: Qwen3-4B attention shape, one 4096-token prompt
SS_STEPS, SS_WIN = 1024, 8          # seal-share run: steps, steps per timed window
# Seal roofline. FP32 work of sealing one 128 x 128 group matrix (an FMA counts 2): the
# 128-point Hadamard transform, 7 add/subtract stages per element; Y * Y, 1; 16 Sinkhorn
# iterations of two matrix-vector passes over Y * Y, 64; the normalised value and its
# grid position (two multiplies and an FMA), 4. 76 FLOP per element.
SEAL_FLOP = 76 * 128 * 128
FP32_LANES_PER_SM = 128


def prefill_leg(torch, device, stream, barrier, reps=5, cpu=False):
    """Prompt prefill: kvarn_prefill (bulk append of 4096 tokens, sealing 31 groups per
    KV head and side, then causal many-query attention of all 4096 queries). Each rep
    starts from an empty sequence; L2 is flushed (a 256 MiB write) before each timed call.
    Also times kvarn_prefill_attention alone on the filled cache for its roofline."""
    from quantized_kv_cache_seal_gb300 import workloads
    from quantized_kv_cache_seal_gb300.cache import KVarNCache

    cache = KVarNCache(num_layers=1, max_seqs=1, num_q_heads=PF_HQ, num_kv_heads=PF_HKV, k_bits=KB, v_bits=VB,
                       tail_floor=FLOOR, max_seq_len=PF_N, device=device)
    k, v = workloads.torch_tokens(SEED + 11, 0, 0, PF_N, PF_HKV, device=device)
    k, v = k.contiguous(), v.contiguous()
    q = workloads.torch_queries(SEED + 12, PF_N, 1, PF_HQ, device=device)[:, 0].contiguous()
    out = torch.empty_like(q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fused, attn = [], []
    for rep in range(reps + 2):  # the first two untimed
        cache.release(0)
        flush.fill_(rep & 255)
        barrier()
        e0.record(stream)
        cache.prefill(0, [0], [PF_N], k, v, q, out)
        e1.record(stream)
        barrier()
        if rep >= 2:
            fused.append(e0.elapsed_time(e1))
        flush.fill_((rep + 1) & 255)
        barrier()
        e0.record(stream)
        cache.prefill_attention(0, [0], [PF_N], q, out)
        e1.record(stream)
        barrier()
        if rep >= 2:
            attn.append(e0.elapsed_time(e1))
    err = cache.check_device_error()
    cache.close()
    if err:
        raise RuntimeError(f"device error word after prefill: {err}")
    f_ms, a_ms = statistics.median(fused), statistics.median(attn)
    flops = PF_HQ * 4 * 128 * (PF_N * (PF_N + 1) / 2)  # causal QK + PV, 2 flops per MAC
    peak, kind = measured_tensor_peak()
    ach = flops / (a_ms * 1e-3) / 1e12
    return {
        "workload": f"qwen3_4b_gqa32x8_prompt{PF_N}_k{KB}v{VB}" + (f"_tail_floor{FLOOR}" if FLOOR else ""),
        "tokens_per_s": PF_N / (f_ms * 1e-3), "fused_ms": f_ms, "attention_ms": a_ms, "append_seal_ms": f_ms - a_ms,
        "l2": "flushed (256 MiB write) before each timed call",
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                     "traffic": profiled_traffic(None, "prefill_kernel_qwen3_4b_prompt4096_k2v2_traffic.json")
                     if FLOOR == 0 and (KB, VB) == (2, 2) else None, "peak_kind": kind, "kernel": f"prefill_kernel<{KB},{VB}>",
                     "alg_flops_per_launch": flops, "launch_us": a_ms * 1e3},
        "gpu_launches_per_prefill": 3,  # seal_jobs_kernel, append_kernel, prefill_kernel
        "cpu_baseline": prefill_cpu_baseline(k.cpu().numpy(), v.cpu().numpy(), q.cpu().numpy(),
                                             positions_sample=256) if cpu else None,
    }


def run_ours(args):
    import torch

    from quantized_kv_cache_seal_gb300 import kvarn as K
    from quantized_kv_cache_seal_gb300 import workloads

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    K_, W = args.steps, args.warmup
    reps_max = max(3, min(args.reps, 8192 // max(K_, 1)))
    total_steps = W + K_ * (reps_max + 2) + SS_STEPS + 8  # timed reps, two e2e passes, seal-share run
    cache, ids, lengths = build_cache(torch, device, total_steps + 256)
    q_all = workloads.torch_queries(SEED + 100 * rank, total_steps, BATCH, HQ, device=device)
    kn_all, vn_all = [], []
    for i in range(BATCH):
        k, v = workloads.torch_tokens(SEED, i, lengths[i], total_steps, HKV, device=device)
        kn_all.append(k)
        vn_all.append(v)
    kn_all = torch.stack(kn_all, 1).contiguous()  # [steps][B][Hkv][d]
    vn_all = torch.stack(vn_all, 1).contiguous()
    out = torch.empty((BATCH, HQ, 128), dtype=torch.float16, device=device)
    stream = torch.cuda.current_stream()
    scale = 1.0 / math.sqrt(128)
    h = cache.handle
    sp = stream.cuda_stream
    cur = [0]
    lens = list(lengths)

    def step():
        s = cur[0]
        K.kvarn_decode_step(h, 0, ids, kn_all[s], vn_all[s], q_all[s], out, scale, sp)
        cur[0] += 1

    def lens_at(s):
        return [n + s for n in lengths]

    for _ in range(W):
        step()
    torch.cuda.synchronize()

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    def run_e2e():
        """e2e and e2e_copies (None, None with --no-e2e); run halfway through the timed
        repetitions, so that the contexts match those of the median repetition."""
        # end to end through the C ABI with host buffers: every step's k, v and q come from
        # pinned host memory and its output goes back to pinned host memory, inside the
        # timed region. Two ways, both reported: (1) the kernels read and write the pinned
        # host buffers themselves (unified addressing; over NVLink-C2C on Grace), used as
        # `e2e` when the library confirms the buffers are device-accessible; (2) explicit
        # copies on a second stream, double buffered (step k + 1 goes up and step k - 1 comes
        # down while step k runs), `e2e_copies`, and `e2e` when (1) is not available.
        e2e, e2e_copies = None, None
        if not args.no_e2e:
            nk, nv, nq = kn_all[0].numel(), vn_all[0].numel(), q_all[0].numel()
            h2d = int((nk + nv + nq) * 2)
            d2h = int(out.numel() * 2)

            def timed(run):
                barrier()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                t_host = time.perf_counter()
                run()
                e1.record(stream)
                t_host = time.perf_counter() - t_host
                barrier()
                ems = max_over_ranks(e0.elapsed_time(e1), pg, device)
                return ems, t_host

            def entry(ems, path):
                return {"value": whole_job_rate(BATCH * K_, world, ems), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "path": path}

            # (1) kernels on the pinned host buffers
            hk = kn_all[cur[0]:cur[0] + K_].cpu().pin_memory()
            hv = vn_all[cur[0]:cur[0] + K_].cpu().pin_memory()
            hq = q_all[cur[0]:cur[0] + K_].cpu().pin_memory()
            hout = torch.empty((K_, BATCH, HQ, 128), dtype=torch.float16).pin_memory()
            mapped = all(K.kvarn_device_accessible(t) for t in (hk, hv, hq, hout))
            if mapped:
                def run_mapped():
                    for k in range(K_):
                        K.kvarn_decode_step(h, 0, ids, hk[k], hv[k], hq[k], hout[k], scale, sp)
                        cur[0] += 1
                ems, t_host = timed(run_mapped)
                e2e = entry(ems, "kernels read and write pinned host buffers")
                print(f"e2e mapped: host loop {t_host / K_ * 1e6:.1f} us per step, device {ems / K_ * 1e3:.1f} us per step",
                      file=sys.stderr)

            # (2) explicit copies, double buffered on a copy stream
            hin = torch.cat([kn_all[cur[0]:cur[0] + K_].reshape(K_, -1), vn_all[cur[0]:cur[0] + K_].reshape(K_, -1),
                             q_all[cur[0]:cur[0] + K_].reshape(K_, -1)], dim=1).cpu().pin_memory()
            cs = torch.cuda.Stream(device=device)
            din = [torch.empty(nk + nv + nq, dtype=torch.float16, device=device) for _ in range(2)]
            dk = [d[:nk].view_as(kn_all[0]) for d in din]
            dv = [d[nk:nk + nv].view_as(vn_all[0]) for d in din]
            dq = [d[nk + nv:].view_as(q_all[0]) for d in din]
            do = [torch.empty_like(out) for _ in range(2)]
            up = [torch.cuda.Event() for _ in range(2)]    # inputs of the buffer set uploaded
            done = [torch.cuda.Event() for _ in range(2)]  # step on the buffer set finished
            down = [torch.cuda.Event() for _ in range(2)]  # output of the buffer set downloaded

            def run_copies():
                cs.wait_stream(stream)
                for k in range(K_):
                    b = k & 1
                    torch.cuda.set_stream(cs)
                    if k >= 2:
                        cs.wait_event(done[b])
                    din[b].copy_(hin[k], non_blocking=True)
                    up[b].record(cs)
                    torch.cuda.set_stream(stream)
                    stream.wait_event(up[b])
                    if k >= 2:
                        stream.wait_event(down[b])
                    K.kvarn_decode_step(h, 0, ids, dk[b], dv[b], dq[b], do[b], scale, sp)
                    done[b].record(stream)
                    torch.cuda.set_stream(cs)
                    cs.wait_event(done[b])
                    hout[k].copy_(do[b], non_blocking=True)
                    down[b].record(cs)
                    torch.cuda.set_stream(stream)
                    cur[0] += 1
                stream.wait_stream(cs)

            ems, t_host = timed(run_copies)
            e2e_copies = entry(ems, "copies on a second stream, double buffered")
            print(f"e2e copies: host loop {t_host / K_ * 1e6:.1f} us per step, device {ems / K_ * 1e3:.1f} us per step",
                  file=sys.stderr)
            if e2e is None:
                e2e = e2e_copies

        return e2e, e2e_copies

    rep_ms, rep_bytes = [], []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    rep = 0
    e2e = e2e_copies = None
    e2e_done = False
    while True:
        if rep == reps_max // 2 and not e2e_done:
            e2e, e2e_copies = run_e2e()
            e2e_done = True
        start = cur[0]
        bytes_rep = sum(step_bytes(lens_at(s)) for s in range(start, start + K_))
        barrier()
        ev0.record(stream)
        for _ in range(K_):
            step()
        ev1.record(stream)
        barrier()
        rep_ms.append(ev0.elapsed_time(ev1))
        rep_bytes.append(bytes_rep)
        rep += 1
        if rep >= reps_max or (rep >= 3 and time.time() - t_begin > args.min_seconds):
            break
    t_end = time.time()
    sampler.stop()
    if not e2e_done:
        e2e, e2e_copies = run_e2e()
    clocks = sampler.summary(t_begin, t_end)
    err = cache.check_device_error()
    if err != 0:
        raise RuntimeError(f"device error word: {err}")
    order = sorted(range(len(rep_ms)), key=lambda i: rep_ms[i])
    mid = order[len(order) // 2]
    ms = max_over_ranks(rep_ms[mid], pg, device)
    ms_per_step = ms / K_
    value = whole_job_rate(BATCH * K_, world, ms)
    launch_us = ms_per_step * 1e3
    alg_bytes = rep_bytes[mid] / K_
    achieved = alg_bytes / (launch_us * 1e-6) / 1e9
    peak, peak_kind = measured_hbm_peak()

    # seal share (fig1.dev "Why it matters" claims 0.18 % latency overhead): SS_STEPS
    # consecutive steps, in which every sequence seals twice at staggered steps, timed back
    # to back in windows of SS_WIN steps (one event pair per window: per-step events break
    # the programmatic launch chain between steps). The number of fused seals per window
    # varies; a least-squares fit of window time on it gives the time one seal adds to its
    # step, and the share is what the run's seals add over the run's time. This is the
    # difference between the run and the same steps with those groups already sealed.
    n_win = SS_STEPS // SS_WIN
    wev = [torch.cuda.Event(enable_timing=True) for _ in range(n_win + 1)]
    seals_w = []
    barrier()
    wev[0].record(stream)
    for wi in range(n_win):
        ns = 0
        for _ in range(SS_WIN):
            ns += sealing_count(lens_at(cur[0]))
            step()
        wev[wi + 1].record(stream)
        seals_w.append(ns)
    barrier()
    tw = [wev[i].elapsed_time(wev[i + 1]) for i in range(n_win)]
    seal_share, seal_steps = None, None
    if len(set(seals_w)) > 1:
        X = np.stack([np.ones(n_win), np.array(seals_w, np.float64)], 1)
        coef, *_ = np.linalg.lstsq(X, np.array(tw, np.float64), rcond=None)
        resid = np.array(tw) - X @ coef
        dof = max(n_win - 2, 1)
        cov = (resid @ resid / dof) * np.linalg.inv(X.T @ X)
        per_seal_ms = float(coef[1])
        seal_share = max(0.0, per_seal_ms * sum(seals_w) / sum(tw))
        seal_steps = {"steps": SS_STEPS, "window": SS_WIN, "seals": int(sum(seals_w)),
                      "us_per_seal": per_seal_ms * 1e3, "us_per_seal_stderr": float(math.sqrt(cov[1, 1])) * 1e3,
                      "us_per_step": sum(tw) / SS_STEPS * 1e3,
                      "method": "window time regressed on fused seals per window; share = fitted seal time / run time"}

    # bulk seal throughput: kvarn_seal_groups on as many group matrices as the headline
    # cache holds (16 sequences x 255 groups x 8 KV heads x K and V = 65,280; 2.1 GB in)
    seal_gps = None
    if not args.no_seal:
        from quantized_kv_cache_seal_gb300.cache import seal_groups
        n = 16 * 255 * 8 * 2
        x, _ = workloads.torch_tokens(SEED + 7, 99, 0, n * 128 // HKV, HKV, device=device)
        x = x.view(n, 128, 128)
        # untimed, at full size: the outputs' allocation is then cached, not timed
        seal_groups(x, 2, 0)
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        seal_groups(x, 2, 0)
        s1.record(stream)
        barrier()
        seal_gps = n / (s0.elapsed_time(s1) / 1e3) * world
        del x

    workloads_res = None if args.no_workloads or (KB, VB, FLOOR) != (2, 2, 0) else workload_leg(
        torch, device, stream, barrier, peak)
    prefill = None if args.no_prefill else prefill_leg(
        torch, device, stream, barrier, cpu=rank == 0 and world == 1 and not args.no_cpu_baseline)
    snapshot = None if args.no_snapshot or world > 1 else snapshot_leg(cache)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K_, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"f16 mma / f32 accum on {KB}/{VB}-bit codes", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": BATCH * world, "seq_len": int(statistics.mean(lengths)),
                   "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": 128, "k_bits": KB, "v_bits": VB,
                   "parallelism": f"replicas{world}", "l2": "working set ~315 MB per step > 129 MB L2 (no flush)",
                   "reps": len(rep_ms), "rep_ms": [round(x, 4) for x in rep_ms]},
        "gpu_launches": 2 * K_,  # per step: the decode kernel and its merge kernel
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": args.traffic if args.traffic is not None else
                     (profiled_traffic(alg_bytes) if FLOOR == 0 and (KB, VB) == (2, 2) else None),
                     "peak_kind": peak_kind, "kernel": f"decode_kernel<{KB},{VB}>",
                     "alg_bytes_per_launch": alg_bytes, "launch_us": launch_us},
        "seal_groups_per_s": seal_gps,
        "seal_roofline": seal_roofline(seal_gps, clocks, torch),
        "workloads": workloads_res,
        "prefill": prefill,
        "snapshot": snapshot,
        "seal_share": seal_share,
        "seal_steps": seal_steps,
        "clocks": clocks,
        "e2e": e2e,
        "e2e_copies": e2e_copies,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cache, lengths, cur[0], q_all, args.cpu_pairs)
    if pg is not None:
        pg.destroy_process_group()
    cache.close()
    if rank == 0:
        print(json.dumps(result), flush=True)


def seal_roofline(seal_gps, clocks, torch):
    """The bulk seal against the FP32 ALU peak of this GPU: SEAL_FLOP per group matrix
    times groups/s, over SMs x 128 FP32 lanes x 2 FLOP per FMA x the SM clock (the
    largest sampled, nvidia-smi's clocks.max.sm, else 2070 MHz)."""
    if not seal_gps:
        return None
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    peak = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    achieved = seal_gps * SEAL_FLOP / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "flop_per_group": SEAL_FLOP, "peak_kind": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x "
                                                      f"{mhz:.0f} MHz", "kernel": "seal_groups_kernel"}


WORKLOAD_LEG = [  # (workload name, steps timed, bit widths); C3 is the headline line itself
    ("c2_qwen3_4b_4k", 256, None),
    ("c4_long_64k_k4v2", 2048, None),
    ("c4_long_64k_k4v4", 2048, None),
    ("c5_phi4_14b_ragged_b2", 64, None),
    ("c5_phi4_14b_ragged_b4", 64, None),
    ("c5_phi4_14b_ragged_b8", 64, None),
]


def workload_leg(torch, device, stream, barrier, peak):
    """The other decode workloads, each through the same kvarn_decode_step loop: the cache
    prefilled by bulk append, a few untimed steps, then its stated number of decode steps
    timed back to back (two passes from the same state, the faster kept). Reported per
    workload: us per step, tokens/s, algorithmic HBM GB/s and the fraction of the
    measured peak (for the single-sequence Qwen3-4B shape the step is launch- and
    latency-bound: its fraction is not a meaningful roofline)."""
    from quantized_kv_cache_seal_gb300 import workloads
    from quantized_kv_cache_seal_gb300 import kvarn as K
    from quantized_kv_cache_seal_gb300.cache import KVarNCache

    wl = workloads.workloads()
    out = {}
    for name, steps, _ in WORKLOAD_LEG:
        w = wl[name]
        lengths = list(w.context)
        warm = 4
        cache = KVarNCache(num_layers=1, max_seqs=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                           k_bits=w.k_bits, v_bits=w.v_bits, max_seq_len=max(lengths) + 2 * (steps + warm),
                           device=device)
        done = [0] * w.batch
        while any(d < n for d, n in zip(done, lengths)):
            ids, counts, ks, vs = [], [], [], []
            for i in range(w.batch):
                c = min(8192, lengths[i] - done[i])
                if c > 0:
                    k, v = workloads.torch_tokens(w.seed, i, done[i], c, w.num_kv_heads, spike_frac=w.spike_frac,
                                                  spike_factor=w.spike_factor, device=device)
                    ids.append(i)
                    counts.append(c)
                    ks.append(k)
                    vs.append(v)
                    done[i] += c
            cache.append(0, ids, counts, torch.cat(ks), torch.cat(vs))
        total = warm + steps
        kn, vn = [], []
        for i in range(w.batch):
            k, v = workloads.torch_tokens(w.seed, i, lengths[i], total, w.num_kv_heads, spike_frac=w.spike_frac,
                                          spike_factor=w.spike_factor, device=device)
            kn.append(k)
            vn.append(v)
        kn = torch.stack(kn, 1).contiguous()
        vn = torch.stack(vn, 1).contiguous()
        qs = workloads.torch_queries(w.seed, total, w.batch, w.num_q_heads, device=device)
        outb = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float16, device=device)
        ids = list(range(w.batch))
        scale = 1.0 / math.sqrt(128)
        h, sp = cache.handle, stream.cuda_stream
        img = cache.snapshot()
        best = None
        for rep in range(2):
            if rep:
                cache.restore(img)
            base = 0
            for k in range(warm):
                K.kvarn_decode_step(h, 0, ids, kn[base + k], vn[base + k], qs[base + k], outb, scale, sp)
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k in range(warm, total):
                K.kvarn_decode_step(h, 0, ids, kn[base + k], vn[base + k], qs[base + k], outb, scale, sp)
            e1.record(stream)
            barrier()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        err = cache.check_device_error()
        cache.close()
        if err:
            raise RuntimeError(f"device error word in {name}: {err}")
        nbytes = sum(step_bytes([n + warm + k for n in lengths], w.num_q_heads, w.num_kv_heads, w.k_bits, w.v_bits)
                     for k in range(steps))
        us = best / steps * 1e3
        gbs = nbytes / (best * 1e-3) / 1e9
        entry = {"steps": steps, "us_per_step": us, "tokens_per_s": w.batch * steps / (best * 1e-3),
                 "hbm_gbs": gbs, "frac": gbs / peak, "alg_bytes_per_step": nbytes / steps,
                 "batch": w.batch, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                 "k_bits": w.k_bits, "v_bits": w.v_bits, "mean_context": int(statistics.mean(lengths))}
        if w.batch == 1:
            entry["note"] = "one sequence: launch- and latency-bound, the roofline fraction is not meaningful"
        out[name] = entry
        del kn, vn, qs, img
        torch.cuda.empty_cache()
    return out


def _oracle_step_sample(cache, q_np, pairs, threads=None):
    """Time the oracle's attention for the given (seq, kv head) pairs on host threads."""
    import concurrent.futures

    import oracle

    jobs = []
    mem = cache.mem.cpu().numpy()
    base = cache.mem.data_ptr()
    from quantized_kv_cache_seal_gb300 import kvarn as K
    for (s, h) in pairs:
        n = cache.length(0, s)
        ng = sealed_groups(n)
        nt = max(n - 128, 0) - 128 * ng
        kr = np.stack([mem[(p - base):(p - base) + nb] for p, nb in
                       (K.kvarn_group_record(cache.handle, 0, s, g, h, 0) for g in range(ng))])
        vr = np.stack([mem[(p - base):(p - base) + nb] for p, nb in
                       (K.kvarn_group_record(cache.handle, 0, s, g, h, 1) for g in range(ng))])
        ring = 128 * (FLOOR + 1)  # tail ring rows; slot = (position - 128) mod ring
        regions = K.kvarn_exact_regions(cache.handle, 0, s)
        sk, sv = [mem[(p - base):(p - base) + HKV * 128 * 128 * 2].view(np.float16).reshape(HKV, 128, 128)
                  for p in regions[:2]]
        tk, tv = [mem[(p - base):(p - base) + HKV * ring * 128 * 2].view(np.float16).reshape(HKV, ring, 128)
                  for p in regions[2:]]
        idx = (128 * ng + np.arange(nt)) % ring
        r = HQ // HKV
        jobs.append((q_np[s, h * r:(h + 1) * r], sk[h], sv[h], kr, vr, tk[h, idx], tv[h, idx]))
    cores = os.cpu_count() or 1

    def one(j):
        q, sk, sv, kr, vr, tk, tv = j
        return oracle.attention(q, 1.0 / math.sqrt(128), sk, sv, kr, vr, tk, tv, KB, VB)

    n_threads = min(threads or cores, len(jobs))
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=n_threads) as ex:
        list(ex.map(one, jobs))
    return time.perf_counter() - t0, n_threads


def cpu_baseline(cache, lengths, s_now, q_all, n_pairs):
    """The oracle timed on this host's cores on a bounded sample of the same workload:
    decode attention for n_pairs (sequence, KV head) pairs of the current cache state."""
    import oracle

    oracle.build()
    q_np = q_all[s_now - 1].cpu().numpy()
    pairs = [(i % BATCH, (i * 3) % HKV) for i in range(n_pairs)]
    t, used = _oracle_step_sample(cache, q_np, pairs)
    step_s = t * (BATCH * HKV) / len(pairs)
    t1, _ = _oracle_step_sample(cache, q_np, pairs[:2], threads=1)  # the oracle on one thread
    single_s = t1 * (BATCH * HKV) / 2
    # oracle seal throughput on 2 * cores group matrices
    from quantized_kv_cache_seal_gb300 import workloads
    import concurrent.futures
    cores = os.cpu_count() or 1
    xs = workloads.group_matrices(SEED + 11, 2 * cores)
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(lambda x: oracle.seal(x, KB, 0), list(xs)))
    seal_gps = len(xs) / (time.perf_counter() - t0)
    return {"value": BATCH / step_s, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"decode attention of {len(pairs)} of {BATCH * HKV} (sequence, KV head) pairs at ~32k "
                      f"context over the cache's records, scaled to the whole step; seal: {len(xs)} group matrices",
            "seal_groups_per_s": seal_gps,
            "single_thread": {"value": BATCH / single_s, "unit": "tokens/s", "cores": 1,
                              "sample": "decode attention of 2 pairs on one thread, scaled to the whole step"}}


def prefill_cpu_baseline(k, v, q, positions_sample=64, head=0):
    """The oracle's prefill attention, as it stands, on this host's cores, on a bounded
    sample of the prompt-prefill leg: one KV head's cache built by the oracle from the
    same tokens (k, v: [n][Hkv][128] fp16 numpy), then the queries of `positions_sample`
    positions spread over the prompt (its r query heads), timed and scaled by the causal
    work (sum over queries of the keys each sees) to the whole prompt and all heads.
    Returns the cpu_baseline object (prompt tokens/s)."""
    import concurrent.futures

    import oracle

    oracle.build()
    n, hkv = k.shape[0], k.shape[1]
    hq = q.shape[1]
    r = hq // hkv
    oc = oracle.OracleCache(1, KB, VB, tail_floor=FLOOR)
    oc.append(0, k[:, head:head + 1], v[:, head:head + 1])  # untimed setup (the oracle's seals)
    st = oc.seqs[0]
    n_sink, n_groups, _ = oc.regions(0)
    kr = np.stack([g[0] for g in st["krec"]]) if n_groups else np.zeros((0,), np.uint8)
    vr = np.stack([g[0] for g in st["vrec"]]) if n_groups else np.zeros((0,), np.uint8)
    tk, tv = oc.tail(0)
    pos = sorted({int(x) for x in np.linspace(0, n - 1, positions_sample)})
    cores = os.cpu_count() or 1
    chunks = [pos[i::cores] for i in range(min(cores, len(pos)))]

    def run(ps):
        oracle.prefill_attention(q[ps, head * r:(head + 1) * r], ps, 1.0 / math.sqrt(128), st["sink_k"][:n_sink, 0],
                                 st["sink_v"][:n_sink, 0], kr, vr, tk[:, 0], tv[:, 0], KB, VB)

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        list(ex.map(run, chunks))
    t = time.perf_counter() - t0
    work_sample = sum(p + 1 for p in pos) * r
    work_all = (n * (n + 1) // 2) * hq
    prompt_s = t * work_all / work_sample
    return {"value": n / prompt_s, "unit": "prompt tokens/s", "cores": len(chunks), "kind": "oracle",
            "sample": f"{len(pos)} query positions x {r} query heads of KV head {head}, scaled by causal work "
                      f"to {n} positions x {hq} heads (the oracle's seals of the prompt are untimed setup)"}


def run_reference(args):
    """The oracle (plain fp64 C) on the host cores, on the headline workload: every step
    appends one token to each of the 128 (sequence, KV head) pairs (sealing when a group
    fills) and attends with their query heads, the pairs spread over one thread per core.
    The whole batch is timed every step (nothing is scaled); beside it, one pair-step
    timed on a single thread."""
    import concurrent.futures

    import oracle
    from quantized_kv_cache_seal_gb300 import workloads

    rank, world, local = dist_info()
    if rank != 0:
        return
    oracle.build()
    cores = os.cpu_count() or 1
    n_pairs = BATCH * HKV if args.ref_pairs <= 0 else max(1, min(BATCH * HKV, args.ref_pairs))
    lengths = c3_lengths()
    pairs = [(i % BATCH, (i // BATCH + 3 * (i % BATCH)) % HKV) for i in range(n_pairs)]
    if n_pairs == BATCH * HKV:
        pairs = [(s, h) for s in range(BATCH) for h in range(HKV)]
    setup0 = time.perf_counter()
    srcs = {s: workloads.TokenSource(SEED, s, HKV) for s in {p[0] for p in pairs}}
    toks = {s: srcs[s].tokens(0, lengths[s] + args.warmup + args.steps + 1) for s in srcs}

    def setup(pair):
        s, h = pair
        oc = oracle.OracleCache(1, KB, VB, tail_floor=FLOOR)
        k, v = toks[s]
        oc.append(0, k[:lengths[s], h:h + 1], v[:lengths[s], h:h + 1])
        return oc

    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        caches = list(ex.map(setup, pairs))
    setup_s = time.perf_counter() - setup0
    r = HQ // HKV
    scale = 1.0 / math.sqrt(128)

    def one_step(idx, step, q):
        s, h = pairs[idx]
        pos = lengths[s] + step
        k, v = toks[s]
        caches[idx].append(0, k[pos:pos + 1, h:h + 1], v[pos:pos + 1, h:h + 1])
        caches[idx].attend(0, q[s, h * r:(h + 1) * r], scale)

    times = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        for step in range(args.warmup + args.steps):
            q = workloads.queries(SEED, step, BATCH, HQ)
            t0 = time.perf_counter()
            list(ex.map(lambda i: one_step(i, step, q), range(n_pairs)))
            if step >= args.warmup:
                times.append(time.perf_counter() - t0)
    # one pair-step on one thread (the oracle's single-thread rate), on a fresh copy of a pair
    step1 = args.warmup + args.steps
    t1 = []
    q1 = workloads.queries(SEED, step1, BATCH, HQ)
    for idx in range(min(3, n_pairs)):
        t0 = time.perf_counter()
        one_step(idx, step1, q1)
        t1.append(time.perf_counter() - t0)
    single_step_s = statistics.median(t1) * BATCH * HKV
    per_step = statistics.mean(times) * (BATCH * HKV) / n_pairs
    value = BATCH / per_step
    whole = n_pairs == BATCH * HKV
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": BATCH, "seq_len": int(statistics.mean(lengths)),
                       "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": 128, "k_bits": KB, "v_bits": VB,
                       "parallelism": "host threads", "setup_s": setup_s},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, n_pairs), "kind": "oracle",
                             "sample": (f"the whole batch every step: all {n_pairs} (sequence, KV head) pairs, "
                                        f"append + seal + attention, timed (not scaled)") if whole else
                                       (f"{n_pairs} of {BATCH * HKV} (sequence, KV head) pairs per step, "
                                        f"append + seal + attention, scaled to the whole batch"),
                             "single_thread": {"value": BATCH / single_step_s, "unit": "tokens/s", "cores": 1,
                                               "sample": "median of 3 single pair-steps on one thread, "
                                                         "times 128 pairs"}},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--reps", type=int, default=20, help="timed repetitions of K steps (median reported)")
    ap.add_argument("--min-seconds", type=float, default=1.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-seal", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-snapshot", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the Qwen3-4B / 64k / Phi-4 decode workloads")
    ap.add_argument("--prefill-only", action="store_true", help="run the prompt-prefill leg alone (one JSON object)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=32)
    ap.add_argument("--ref-pairs", type=int, default=0, help="reference arm: pairs per step (0: the whole batch)")
    ap.add_argument("--k-bits", type=int, default=2, help="K code width (the headline workload: 2)")
    ap.add_argument("--v-bits", type=int, default=2, help="V code width (the headline workload: 2)")
    ap.add_argument("--tail-floor", type=int, default=0,
                    help="keep this many full groups exact beyond the partial one (BeeLlama: 1); "
                         "the headline workload is the published design, 0")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the decode kernel, if captured for this build")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global FLOOR, WORKLOAD, KB, VB
    if (args.k_bits, args.v_bits) != (KB, VB):
        KB, VB = args.k_bits, args.v_bits
        WORKLOAD = WORKLOAD.replace("_k2v2", f"_k{KB}v{VB}")
    if args.tail_floor:
        FLOOR = args.tail_floor
        WORKLOAD = f"{WORKLOAD}_tail_floor{FLOOR}"
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        import torch

        torch.cuda.set_device(0)
        res = prefill_leg(torch, torch.device("cuda", 0), torch.cuda.current_stream(), torch.cuda.synchronize)
        print(json.dumps({"prefill": res}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
