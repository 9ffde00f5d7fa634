"""Benchmark of the USP attention hot path (one JSON line on rank 0).

A step is one full pass of the path over one synthetic batch:
  positions/documents -> seq->head all-to-all with RoPE (Q,K) and plain (V),
  padding rows written as zeros -> causal GQA attention forward
  -> head->seq (O) -> seq->head (dO) -> attention backward
  -> head->seq (dQ, dK with inverse RoPE; dV).
The default workload is the 120 000-token SP8 layer (Hq/Hkv/D = 32/8/128,
YaRN RoPE to 131 072).  Inputs (0.98 GB for Q alone) are larger than L2, so
no flush is needed between steps.  The permutation stages' GB/s is taken
from a separate leg that runs each stage alone after a memset of twice the
L2 size.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle, timed

Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
path has no cross-GPU step here, so every rank runs the same workload and
`value` is the tokens of all ranks over the slowest rank's time.
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

METRIC = "USP attn fwd+bwd tokens/s and TFLOP/s (% bf16 peak); repack GB/s (% HBM)"
FLUSH_ITERS = 10        # timed calls of each permutation stage after an L2 flush
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if isinstance(v, (int, float)):
                    out[k] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "ulysses_sequence_attention_usp_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


BWD_SOURCES = ["attn_bwd_tc.cu", "tc_ptx.cuh", "usp_common.cuh"]


def measured_traffic(workload):
    """DRAM bytes per usp_attn_bwd call from the committed ncu summary, or
    None when the kernels changed since those counters were taken."""
    p = os.path.join(ROOT, "profiles", "attn_bwd_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("workload") != workload or d.get("source_sha256") != kernel_source_hash(BWD_SOURCES):
        return None
    return d.get("dram_bytes_per_call")


def reduce_max(value, world, device=None):
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(world, tokens_per_rank, steps, seconds):
    """Whole-job tokens/s: every rank runs the same workload (replicas), so
    the job processes world * tokens * steps tokens in the slowest rank's
    time."""
    return world * tokens_per_rank * steps / seconds


def attended_pairs(S, cu, causal=True):
    """(query, key) pairs attended: per document L(L+1)/2 causal, L^2
    bidirectional."""
    lens = np.array([S], np.int64) if cu is None else np.diff(np.asarray(cu, np.int64))
    return int((lens * (lens + 1) // 2).sum()) if causal else int((lens * lens).sum())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def _query_once(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=30).stdout
        except Exception:
            return []
        return [ln.strip() for ln in out.splitlines() if ln.strip()]

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        res = self._summary(self.lines)
        if res is None:   # the region ended before the first sample: read once right after
            res = self._summary(self._query_once())
            if res is not None:
                res["samples"] = 0
                res["note"] = "timed region shorter than one 200 ms sample; read right after it"
        return res

    @staticmethod
    def _summary(lines):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_bus_id(torch):
    try:
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(wl, inp, target_s, fixed_rows=None, causal=True, keep=False):
    """Time the oracle's forward+backward of query head 0 (and its KV head)
    on the first S' rows, S' grown until one run takes about target_s
    seconds (or S' = fixed_rows).  Returns (seconds, S', scale factor to the
    full workload), and with keep=True also the last run's results."""
    from oracle import usp_oracle as O
    D = wl.D
    scale = 1.0 / math.sqrt(D)
    cos, sin = O.rope_cos_sin(max(wl.table_len, wl.S), D, wl.rope_base, wl.yarn_factor,
                              wl.yarn_orig_ctx)
    Sp = fixed_rows or 512
    while True:
        Sp = min(Sp, wl.S)
        q = O.bf16_to_f64(inp.q[:Sp, :1])
        k = O.bf16_to_f64(inp.k[:Sp, :1])
        v = O.bf16_to_f64(inp.v[:Sp, :1])
        do = O.bf16_to_f64(inp.do[:Sp, :1])
        cu = None
        if inp.cu is not None:
            cu = np.concatenate([inp.cu[inp.cu < Sp], [Sp]]).astype(np.int64)
        t0 = time.perf_counter()
        res = O.full_sequence(q, k, v, do, cu, cos, sin, scale, causal)
        dt = time.perf_counter() - t0
        if fixed_rows or dt >= target_s / 3 or Sp >= wl.S:
            break
        Sp = int(Sp * min(4.0, max(1.3, math.sqrt(target_s / max(dt, 1e-3)))))
    pairs_s = attended_pairs(Sp, cu, causal)
    pairs_f = attended_pairs(wl.S, inp.cu, causal)
    factor = (pairs_f * wl.Hq) / pairs_s
    return (dt, Sp, factor, res) if keep else (dt, Sp, factor)


def parity_sample(ua, wl, ref, Sp):
    """The GPU step's O, LSE and dQ of query head 0 on rows [0, S') against
    the oracle run of the CPU-baseline leg.  With causal attention those rows
    see only keys below S', so the oracle's values there are the full
    problem's; the oracle rotates exactly in fp64, the GPU by the fp32 table
    into bf16, so LSE differs by the rounding of the rotated Q, K."""
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    o, dq = f(ua.o[:Sp, 0]), f(ua.dq[:Sp, 0])
    lse = ua.lse.reshape(wl.Hq, -1)[0, :Sp].cpu().numpy().astype(np.float64)
    ro, rdq, rl = ref["o"][:, 0], ref["dq"][:, 0], ref["lse"][0]
    d_o, d_dq = np.abs(o - ro), np.abs(dq - rdq)
    fin = np.isfinite(rl)
    res = {"sample": f"query head 0, rows [0, {Sp}) of the timed workload",
           "o_max_abs": float(d_o.max()), "o_mean_abs": float(d_o.mean()),
           "dq_max_rel": float(d_dq.max() / max(float(np.abs(rdq).max()), 1e-30)),
           "lse_max_abs": float(np.abs(lse[fin] - rl[fin]).max()) if fin.any() else 0.0,
           "criteria": {"o_max_abs": 2e-2, "o_mean_abs": 2e-3, "dq_max_rel": 5e-2}}
    res["within_criteria"] = (res["o_max_abs"] <= 2e-2 and res["o_mean_abs"] <= 2e-3
                              and res["dq_max_rel"] <= 5e-2)
    return res


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def l2_note(step_in_bytes, l2_bytes):
    """How L2 is treated by the timing, for the bench line's config."""
    if step_in_bytes > l2_bytes:
        step = ("step: inputs larger than L2 (%.2f GB of Q, K, V, dO), no flush"
                % (step_in_bytes / 1e9))
    else:
        step = ("step: inputs smaller than L2 (%.1f MB of Q, K, V, dO), not flushed "
                "between steps" % (step_in_bytes / 1e6))
    return step + ("; repack GB/s: each stage timed alone after a %d MB memset"
                   % (2 * l2_bytes >> 20))


def workload_config(args, wl, world=1):
    """The `config` keys both arms print for the same flags."""
    allgather = args.cp == "allgather"
    return {"workload": wl.name, "S": wl.S, "P": wl.P, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
            "rope": ("yarn x%g to %d" % (wl.yarn_factor, wl.rope_len)
                     if wl.yarn_factor > 1 else "base %g" % wl.rope_base),
            "attention": "bidirectional" if args.bidirectional else "causal",
            "shards": ("contiguous, K/V all-gather context parallelism"
                       if allgather else "zigzag" if args.zigzag else "contiguous"),
            "ring": args.ring,
            "launch": "CUDA graph replay" if getattr(args, "graph", False) else "eager",
            "parallelism": (f"replicas x{world} (P={wl.P} virtual CP ranks per GPU)"
                            if allgather else
                            f"replicas x{world} (P={wl.P} virtual shards per GPU)")}


def base_line(args, wl, world, value, ms_per_step, dtype):
    """The keys both arms print, with the same `config` for the same flags."""
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": workload_config(args, wl, world)}


def run_reference(args, wl, inp):
    """--impl reference: the oracle, timed on host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    times, raw = [], []
    causal = not args.bidirectional
    _, Sp, factor = oracle_sample(wl, inp, args.ref_seconds, causal=causal)
    for i in range(args.warmup + args.steps):
        dt, Sp, factor = oracle_sample(wl, inp, args.ref_seconds, fixed_rows=Sp, causal=causal)
        if i >= args.warmup:
            times.append(dt * factor)
            raw.append(dt)
    full_s = statistics.median(times)
    value = wl.S / full_s
    sample = (f"oracle fwd+bwd of q head 0 / kv head 0 on the first {Sp} rows, "
              f"scaled by attended pairs x heads ({factor:.4g}x) to the full workload")
    line = dict(impl="reference", **base_line(args, wl, args.gpus, value, full_s * 1e3, "f64"))
    line.update({
        # a step is a bounded sample of the workload; its time is scaled up
        "ms_per_step_extrapolated": True,
        "ms_per_step_basis": (f"median over {args.steps} steps of the oracle's time on the "
                              f"sample ({statistics.median(raw) * 1e3:.0f} ms) x {factor:.4g}"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    })
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_usp(args, wl, inp):
    import torch
    import torch.distributed as dist
    from ulysses_sequence_attention_usp_gb300 import build as _build
    _build.build()
    from ulysses_sequence_attention_usp_gb300 import binding as B
    from ulysses_sequence_attention_usp_gb300.pipeline import (AllGatherCPAttention,
                                                               UlyssesAttention)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    causal = not args.bidirectional
    allgather = args.cp == "allgather"

    def make_pipeline(rope_table=None):
        if allgather:
            return AllGatherCPAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                                        rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                                        yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len,
                                        device=dev, rope_table=rope_table, causal=causal)
        return UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                                rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                                yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len, device=dev,
                                rope_table=rope_table, causal=causal, zigzag=args.zigzag,
                                ring=args.ring)

    ua = make_pipeline()
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    st = torch.cuda.current_stream(dev)
    if args.graph:   # graph capture needs a stream other than the default one
        st = torch.cuda.Stream(dev)
        st.wait_stream(torch.cuda.current_stream(dev))
    d = ua.dims
    rows = getattr(ua, "S_pad", wl.S)          # rows of the sequence-layout buffers
    bq = rows * wl.Hq * wl.D * 2
    bkv = rows * wl.Hkv * wl.D * 2
    tab = rows * wl.D * 4                      # one (cos, sin) row per position

    # the stages of one step, in order (all on `st`), and the algorithmic
    # bytes of the permutation / RoPE stages
    if allgather:
        stages = [
            ("positions", lambda: B.usp_pad_shard(d, None, 0, None, ua.pos, ua.doc, st)),
            ("rope_qk", lambda: (
                B.usp_seq_to_head_rope(d, q, wl.Hq, ua.pos, ua.rope, ua.rope_len, 1, ua.q_r, st),
                B.usp_seq_to_head_rope(d, k, wl.Hkv, ua.pos, ua.rope, ua.rope_len, 1, ua.k_r,
                                       st))),
            ("attn_fwd", lambda: B.usp_attn_fwd(d, ua.q_r, ua.k_r, v, ua.doc, ua.o, ua.lse, st)),
            ("attn_bwd", lambda: B.usp_attn_bwd(d, ua.q_r, ua.k_r, v, ua.o, ua.lse, do, ua.doc,
                                                ua.dq_r, ua.dk_r, ua.dv, ua.ws, ua.ws_bytes,
                                                st)),
            ("rope_grads", lambda: (
                B.usp_head_to_seq(d, ua.dq_r, wl.Hq, ua.pos, ua.rope, ua.rope_len, -1, ua.dq,
                                  st),
                B.usp_head_to_seq(d, ua.dk_r, wl.Hkv, ua.pos, ua.rope, ua.rope_len, -1, ua.dk,
                                  st))),
        ]
        rep_bytes = {"rope_qk": 2 * (bq + bkv) + 2 * tab, "rope_grads": 2 * (bq + bkv) + 2 * tab}
    else:
        # the same calls as UlyssesAttention.forward/backward: in the
        # contiguous layout the all-to-all reads the unpadded inputs and
        # writes padding rows as zeros, so the first stage only emits
        # positions and documents; zigzag shards are padded copies first
        if args.zigzag:
            src = (ua.q_seq, ua.k_seq, ua.v_seq, ua.do_seq)
            first = ("pad_qkv", lambda: (
                B.usp_pad_shard(d, q, wl.Hq, ua.q_seq, ua.pos, ua.doc, st),
                B.usp_pad_shard(d, k, wl.Hkv, ua.k_seq, None, None, st),
                B.usp_pad_shard(d, v, wl.Hkv, ua.v_seq, None, None, st)))
        else:
            src = (q, k, v, do)
            first = ("positions", lambda: B.usp_pad_shard(d, None, 0, None, ua.pos, ua.doc, st))
        stages = [
            first,
            ("repack_qkv", lambda: (
                B.usp_seq_to_head_rope(d, src[0], wl.Hq, ua.pos, ua.rope, ua.rope_len, 1,
                                       ua.q_h, st),
                B.usp_seq_to_head_rope(d, src[1], wl.Hkv, ua.pos, ua.rope, ua.rope_len, 1,
                                       ua.k_h, st),
                B.usp_seq_to_head_rope(d, src[2], wl.Hkv, None, None, 0, 0, ua.v_h, st))),
            ("attn_fwd", lambda: ua.attention_forward(st)),     # one launch, or the ring steps
            ("repack_o", lambda: B.usp_head_to_seq(d, ua.o_h, wl.Hq, None, None, 0, 0, ua.o, st)),
        ]
        if args.zigzag:
            stages.append(("pad_do", lambda: B.usp_pad_shard(d, do, wl.Hq, ua.do_seq, None, None,
                                                             st)))
        stages += [
            ("repack_do", lambda: B.usp_seq_to_head_rope(d, src[3], wl.Hq, None, None, 0, 0,
                                                         ua.do_h, st)),
            ("attn_bwd", lambda: B.usp_attn_bwd(d, ua.q_h, ua.k_h, ua.v_h, ua.o_h, ua.lse,
                                                ua.do_h, ua.doc, ua.dq_h, ua.dk_h, ua.dv_h,
                                                ua.ws, ua.ws_bytes, st)),
            ("repack_grads", lambda: (
                B.usp_head_to_seq(d, ua.dq_h, wl.Hq, ua.pos, ua.rope, ua.rope_len, -1, ua.dq,
                                  st),
                B.usp_head_to_seq(d, ua.dk_h, wl.Hkv, ua.pos, ua.rope, ua.rope_len, -1, ua.dk,
                                  st),
                B.usp_head_to_seq(d, ua.dv_h, wl.Hkv, None, None, 0, 0, ua.dv, st))),
        ]
        rep_bytes = {"repack_qkv": 2 * (bq + 2 * bkv) + 2 * tab, "repack_o": 2 * bq,
                     "repack_do": 2 * bq, "repack_grads": 2 * (bq + 2 * bkv) + 2 * tab}
    stage_names = [n for n, _ in stages]
    n_marks = len(stages) + 1

    def step(ev=None):
        for j, (_, call) in enumerate(stages):
            if ev is not None:
                ev[j].record(st)
            call()
        if ev is not None:
            ev[len(stages)].record(st)

    for _ in range(args.warmup):
        step()
    ua.check(st)
    graph, per_step = None, 0
    if args.graph:   # one step's launches, recorded once and replayed
        graph = torch.cuda.CUDAGraph()
        n0 = B.usp_launch_count()
        with torch.cuda.stream(st):
            graph.capture_begin(capture_error_mode="thread_local")
            try:
                step()
            finally:
                graph.capture_end()
        per_step = B.usp_launch_count() - n0
        with torch.cuda.stream(st):
            graph.replay()
        ua.check(st)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_marks)]
           for _ in range(args.steps)]
    clocks = ClockSampler(gpu_bus_id(torch))
    clocks.start()
    barrier()
    n0 = B.usp_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(st)
    if graph is not None:
        with torch.cuda.stream(st):
            for i in range(args.steps):
                graph.replay()
    else:
        for i in range(args.steps):
            step(evs[i])
    t_end.record(st)
    barrier()
    launches = B.usp_launch_count() - n0 + per_step * (args.steps if graph is not None else 0)
    clk = clocks.stop()
    ua.check(st)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    if graph is not None:   # per-stage times from the same steps run eagerly
        for i in range(args.steps):
            step(evs[i])
        barrier()
        ua.check(st)
    stage_ms = {n: statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, n in enumerate(stage_names)}
    elapsed = reduce_max(elapsed, world, dev)

    # ---- the permutation stages alone, each preceded by a memset of twice
    # the L2 size so that none of its inputs is L2-resident: their GB/s is
    # then HBM bandwidth.  Median of FLUSH_ITERS calls of each stage.
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20)
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    rep_calls = {n: c for n, c in stages if n in rep_bytes}
    flushed_ms = {}
    with torch.cuda.stream(st):
        for name, call in rep_calls.items():
            times = []
            for _ in range(FLUSH_ITERS):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                call()
                e1.record(st)
                times.append((e0, e1))
            st.synchronize()
            flushed_ms[name] = statistics.median(a.elapsed_time(b) for a, b in times)
    ua.check(st)
    del flush

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs host->device (one copy stream), runs the step (`st`)
    # and copies its O, dQ, dK, dV device->host (another copy stream).  Two
    # pipelines with their own device buffers alternate, so the copies of
    # one step overlap the compute of its neighbours; events order a
    # pipeline's reuse after its previous step's copies.
    pin = lambda a: torch.from_numpy(a.view(np.int16)).pin_memory()  # noqa: E731
    h_in = [pin(inp.q), pin(inp.k), pin(inp.v), pin(inp.do)]
    ua2 = make_pipeline(ua.rope_host)
    pipes = [(ua, (q, k, v, do)), (ua2, tuple(torch.empty_like(t) for t in (q, k, v, do)))]
    h_out = [[torch.empty(t.shape, dtype=torch.int16).pin_memory()
              for t in (ua.o, ua.dq, ua.dk, ua.dv)] for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_free = [None, None]      # compute of the pipeline's last step finished
    out_read = [None, None]     # its outputs were copied to the host

    def e2e_step(i):
        a, ins = pipes[i % 2]
        if in_free[i % 2] is not None:
            s_h2d.wait_event(in_free[i % 2])
        with torch.cuda.stream(s_h2d):          # Q, K, V first: the forward needs only them
            for src, dst in zip(h_in[:3], ins[:3]):
                dst.view(torch.int16).copy_(src, non_blocking=True)
        ev_qkv = torch.cuda.Event()
        ev_qkv.record(s_h2d)
        with torch.cuda.stream(s_h2d):
            ins[3].view(torch.int16).copy_(h_in[3], non_blocking=True)
        ev_do = torch.cuda.Event()
        ev_do.record(s_h2d)
        st.wait_event(ev_qkv)
        if out_read[i % 2] is not None:
            st.wait_event(out_read[i % 2])
        a.forward(*ins[:3], st)
        ev_fwd = torch.cuda.Event()
        ev_fwd.record(st)
        st.wait_event(ev_do)
        a.backward(ins[3], st)
        done = torch.cuda.Event()
        done.record(st)
        in_free[i % 2] = done
        outs = (a.o, a.dq, a.dk, a.dv)
        s_d2h.wait_event(ev_fwd)                 # O goes down while the backward runs
        with torch.cuda.stream(s_d2h):
            h_out[i % 2][0].copy_(outs[0].view(torch.int16), non_blocking=True)
        s_d2h.wait_event(done)
        with torch.cuda.stream(s_d2h):
            for src, dst in zip(outs[1:], h_out[i % 2][1:]):
                dst.copy_(src.view(torch.int16), non_blocking=True)
        ev_out = torch.cuda.Event()
        ev_out.record(s_d2h)
        out_read[i % 2] = ev_out

    for i in range(2):
        e2e_step(i)
    barrier()
    a_ev = torch.cuda.Event(enable_timing=True)
    b_ev = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(4, args.steps)      # the first upload and the last download are not hidden
    a_ev.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    b_ev.record(s_d2h)
    barrier()
    ua.check(st)
    e2e_t = reduce_max(a_ev.elapsed_time(b_ev) / 1e3, world, dev)
    h2d = sum(a.nbytes for a in (inp.q, inp.k, inp.v, inp.do))
    d2h = sum(t.numel() * 2 for t in (ua.o, ua.dq, ua.dk, ua.dv))
    del ua2, pipes, h_out

    if rank == 0:
        peaks, src = load_peaks()
        pairs = attended_pairs(wl.S, inp.cu, causal)
        f_fwd = 4.0 * wl.D * wl.Hq * pairs
        f_bwd = 10.0 * wl.D * wl.Hq * pairs
        step_s = elapsed / args.steps
        value = aggregate_throughput(world, wl.S, args.steps, elapsed)
        t_fwd = stage_ms["attn_fwd"] / 1e3
        t_bwd = stage_ms["attn_bwd"] / 1e3
        rep_t = sum(stage_ms[n] for n in rep_bytes) / 1e3
        rep_gbs_step = sum(rep_bytes.values()) / rep_t / 1e9
        rep_tf = sum(flushed_ms[n] for n in rep_bytes) / 1e3
        rep_gbs = sum(rep_bytes.values()) / rep_tf / 1e9
        f_bwd_strict = 8.0 * wl.D * wl.Hq * pairs
        peak_t = peaks["bf16_tflops_sustained"]
        bwd_tf = f_bwd / t_bwd / 1e12
        line = base_line(args, wl, world, value, step_s * 1e3, "bf16")
        line.update({
            "l2": l2_note(2 * (bq + bkv), l2),
            "roofline": {"kernel": "usp_attn_bwd (delta + dK/dV + dQ kernels)",
                         "bound": "tensor", "achieved": bwd_tf,
                         "peak": peak_t, "unit": "TFLOP/s", "frac": bwd_tf / peak_t,
                         "traffic": (measured_traffic(wl.name)
                                     if causal and not allgather else None),
                         "peak_source": f"{src} (sustained bf16)",
                         "flops_per_launch": f_bwd},
            "attention": {"fwd_tflops": f_fwd / t_fwd / 1e12, "bwd_tflops": bwd_tf,
                          "fwd_frac": f_fwd / t_fwd / 1e12 / peak_t,
                          "fwd_bwd_tflops": (f_fwd + f_bwd) / (t_fwd + t_bwd) / 1e12,
                          "bwd_tflops_strict": f_bwd_strict / t_bwd / 1e12,
                          "bwd_flops": {"convention_2.5x": f_bwd, "strict_no_recompute": f_bwd_strict},
                          "fwd_ms": t_fwd * 1e3, "bwd_ms": t_bwd * 1e3,
                          "attended_pairs": pairs},
            "repack": {"stages": list(rep_bytes), "gbps": rep_gbs,
                       "frac": rep_gbs / peaks["hbm_gbs"],
                       "peak_gbps": peaks["hbm_gbs"], "peak_source": src,
                       "bytes_per_step": sum(rep_bytes.values()),
                       "timing": "each stage alone, L2 flushed before each call, "
                                 "median of %d" % FLUSH_ITERS,
                       "stage_ms_l2_flushed": flushed_ms,
                       "gbps_in_step": rep_gbs_step},
            "stage_ms": stage_ms,
            "gpu_launches": launches,
            "e2e": {"value": aggregate_throughput(world, wl.S, e2e_steps, e2e_t), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "copies": "pinned host buffers; copy streams overlap the neighbouring "
                              "steps' compute (two pipelines); Q/K/V go up before dO, O "
                              "comes down during the backward"},
            "clocks": clk,
        })
        if world == 1 and not args.no_cpu_baseline:
            dt, Sp, factor, ref = oracle_sample(wl, inp, args.cpu_seconds, causal=causal,
                                                keep=True)
            line["cpu_baseline"] = {
                "value": wl.S / (dt * factor), "unit": "tokens/s", "cores": cpu_cores(),
                "kind": "oracle",
                "sample": (f"oracle fwd+bwd of q head 0 / kv head 0 on the first {Sp} rows "
                           f"({dt:.1f} s), scaled by attended pairs x heads ({factor:.4g}x)")}
            # the same oracle run against the GPU's outputs on those rows (rows
            # in sequence order: not for the zigzag layout; causal only)
            if causal and not args.zigzag:
                line["parity"] = parity_sample(ua, wl, ref, Sp)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="usp", choices=["usp", "reference"])
    ap.add_argument("--workload", default="sp8_120k")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bidirectional", action="store_true",
                    help="attention over the whole document (causal = 0)")
    ap.add_argument("--zigzag", action="store_true",
                    help="zigzag shard layout (rank r holds chunks r and 2P-1-r of 2P)")
    ap.add_argument("--ring", type=int, default=1,
                    help="ring steps of the forward (key windows merged by log-sum-exp)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one CUDA graph of the step (launch-bound small "
                         "problems); per-stage times then come from eager steps")
    ap.add_argument("--cp", choices=["ulysses", "allgather"], default="ulysses",
                    help="sequence parallelism: Ulysses all-to-all (default) or context "
                         "parallelism with a K/V all-gather")
    args = ap.parse_args()
    if args.cp == "allgather" and (args.zigzag or args.ring != 1):
        ap.error("--cp allgather runs contiguous shards without ring steps")
    from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, make_inputs
    wl = WORKLOADS[args.workload]
    if args.impl == "reference" and int(os.environ.get("RANK", "0")) != 0:
        return
    inp = make_inputs(wl, 0)
    if args.impl == "reference":
        run_reference(args, wl, inp)
    else:
        run_usp(args, wl, inp)


if __name__ == "__main__":
    main()
