"""Benchmark of the prefix-shared KV attention path on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole path over one batch of synthetic input: the
KV store of the step's new tokens, then the attention the workload needs
(decode with its decode plan, and/or extend).  Inputs are resident in HBM
before timing starts; between timed steps a 256 MiB buffer is written, so that
no KV survives in L2 (129 MB), and a second 256 MiB buffer is read, so that the
lines the write left dirty are written back before the step rather than
inside it; each step is timed with CUDA events on the launching stream.  The decode plan is built once, before timing, from the
host copy of req_to_token (the sharing structure is fixed for the batch).

Workloads (default: few_shot_decode, the configuration the headline metric
is quoted on):
  few_shot_decode         64 x (1024 shared + 256 private + 1), MHA 32x128, 2M slots
  tree_of_thought_decode  256 leaves of a depth-4 fanout-4 tree, GQA 32/8
  cached_prefix_extend    32 x (2048 cached + 512 new), GQA 32/8
  mixed_chat              16 decode x 32k + 16 extend x (4096 + 1024), 64/8
  tiny_extend             4 x (64 cached + 16 new), 4 heads, head_dim 64
  constrained_decode      one compressed-FSM decoding step (masked argmax and
                          jump) for 256 requests over a 128,256-id vocabulary
                          under a JSON-object constraint

One JSON line is printed by rank 0.  Under torchrun every rank runs the same
workload on its own GPU (independent replicas, no collective on the data
path); value = work of all ranks / the slowest rank's time.

--impl reference times the fp64 oracle (the plain CPU definition) on the host
cores, on a bounded sample of the same workload, in the same units.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from prefix_shared_kv_radixattention_gb300 import inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DECODE_KINDS = ("few_shot_decode", "tree_of_thought_decode")
EXTEND_KINDS = ("cached_prefix_extend", "tiny_extend")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, busy_from: int = 0):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), hw=parts[5], hwt=parts[6],
                                 swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------


class GpuStep:
    """Device state of one workload and the step that runs the path on it."""

    def __init__(self, prob: inputs.Problem, torch, rx, extend_path: str = "staged", rope_base: float = 0.0,
                 kv_fp8: bool = False):
        self.torch, self.rx, self.prob = torch, rx, prob
        dev = "cuda"
        p = prob

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        self.k_pool = torch.empty((p.num_slots, p.hkv, p.d), dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.empty_like(self.k_pool)
        idx = torch.from_numpy(p.cached_slots.astype(np.int64)).to(dev)
        for pool, src in ((self.k_pool, p.cached_k), (self.v_pool, p.cached_v)):
            for s in range(0, len(idx), 1 << 16):
                pool.index_copy_(0, idx[s:s + (1 << 16)], bf(src[s:s + (1 << 16)]))
        self.rtt = i32(p.req_to_token)
        self.k_new, self.v_new, self.slots = bf(p.new_k), bf(p.new_v), i32(p.new_slots)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.has_dec = len(p.dec_req_idx) > 0
        self.has_ext = len(p.ext_req_idx) > 0
        self.launches = 1
        if self.has_dec:
            B = len(p.dec_req_idx)
            self.q_dec = bf(p.q_dec)
            self.o_dec = torch.empty_like(self.q_dec)
            self.dec_req, self.dec_len = i32(p.dec_req_idx), i32(p.dec_seq_len)
            self.max_len = int(p.dec_seq_len.max())
            buf, info = rx.rx_decode_plan_build(p.req_to_token, p.dec_req_idx, p.dec_seq_len, p.hq, p.hkv)
            self.plan_info = info
            self.plan = rx.plan_to_device(buf, info, B)
            ws = rx.rx_attn_decode_workspace(B, p.hq, p.hkv, p.d, self.max_len, self.plan)
            self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev) if ws else None
            # per-head kernel (items of several requests), all-heads kernel
            # (single-request items: one q head per kv head, or 8 kv heads
            # with 2 to 16 q heads each), merge of splits
            G = p.hq // p.hkv
            all_heads = (G == 1 and p.hq in (8, 16, 32, 64)) or \
                (p.hkv == 8 and G in (2, 4, 8, 16) and p.hq * p.d * 2 <= 16384)
            n_wide = info.n_wide if all_heads else 0
            self.launches += ((info.n_items - n_wide) > 0) + (n_wide > 0) + (info.max_parts > 1)
            self.decode_kernels = ((["decode_kernel"] if info.n_items - n_wide > 0 else []) +
                                   ([("decode_wide_kernel" if G == 1 else "decode_gqa_kernel")] if n_wide else []) +
                                   (["merge_kernel"] if info.max_parts > 1 else []))
        if self.has_ext:
            self.q_ext = bf(p.q_ext)
            self.o_ext = torch.empty_like(self.q_ext)
            self.qo, self.ext_req = i32(p.qo_indptr), i32(p.ext_req_idx)
            self.ext_P, self.ext_E = i32(p.ext_prefix_len), i32(p.ext_extend_len)
            self.max_E = int(p.ext_extend_len.max())
            self.launches += 1
            self.ext_ws = None
            if extend_path == "staged":
                ctx = int((p.ext_prefix_len + p.ext_extend_len).sum())
                nb = rx.rx_attn_extend_workspace(ctx, len(p.ext_req_idx), p.hkv, p.d)
                self.ext_ws = torch.empty(nb, dtype=torch.uint8, device=dev)
                self.launches += 2  # packed-row offsets + row copy
        # FP8 pools (optional): the step's rows also stored as E4M3 codes
        self.kv_fp8 = kv_fp8
        if kv_fp8:
            self.k8 = torch.zeros((p.num_slots, p.hkv, p.d), dtype=torch.uint8, device=dev)
            self.v8 = torch.zeros_like(self.k8)
            self.launches += 1
        # rotary position embedding (optional): K rotated on its way into the
        # pool, the step's q rows rotated in place
        self.rope_base = rope_base
        if rope_base:
            pos_of = {}
            for r in range(p.req_to_token.shape[0]):
                for j, sl in enumerate(p.req_to_token[r]):
                    if sl >= 0:
                        pos_of[int(sl)] = j
            self.pos_new = i32(np.array([pos_of[int(sl)] for sl in p.new_slots], np.int32))
            if self.has_ext:
                self.pos_ext = i32(np.concatenate([np.arange(P, P + E, dtype=np.int32) for P, E in
                                                   zip(p.ext_prefix_len, p.ext_extend_len)]))
                self.launches += 1
            if self.has_dec:
                self.pos_dec = i32(p.dec_seq_len - 1)
                self.launches += 1

    def kv_store(self):
        if self.rope_base:
            self.rx.rx_kv_store_rope(self.k_pool, self.v_pool, self.k_new, self.v_new, self.slots, self.pos_new,
                                     self.rope_base, self.status)
        else:
            self.rx.rx_kv_store(self.k_pool, self.v_pool, self.k_new, self.v_new, self.slots, self.status)

    def rope_q(self):
        if self.has_ext:
            self.rx.rx_rope(self.q_ext, self.pos_ext, self.rope_base)
        if self.has_dec:
            self.rx.rx_rope(self.q_dec, self.pos_dec, self.rope_base)

    def decode(self):
        p = self.prob
        self.rx.rx_attn_decode(self.k_pool, self.v_pool, self.q_dec, self.o_dec, None, self.dec_req,
                               self.dec_len, self.rtt, self.max_len, p.sm_scale, self.plan, self.ws,
                               self.status)

    def extend(self):
        p = self.prob
        self.rx.rx_attn_extend(self.k_pool, self.v_pool, self.q_ext, self.o_ext, None, self.qo,
                               self.ext_req, self.ext_P, self.ext_E, self.rtt, self.max_E, p.sm_scale,
                               self.status, workspace=self.ext_ws)

    def store_fp8(self):
        self.rx.rx_kv_store_fp8(self.k8, self.v8, 1.0, 1.0, self.k_new, self.v_new, self.slots, self.status)

    def parts(self):
        return [("store", self.kv_store)] + ([("store_fp8", self.store_fp8)] if self.kv_fp8 else []) + \
            ([("rope_q", self.rope_q)] if self.rope_base else []) + \
            ([("extend", self.extend)] if self.has_ext else []) + ([("decode", self.decode)] if self.has_dec else [])

    def capture(self):
        """Captures each part of the step (after warm-up) as a CUDA graph;
        replaying one runs the same kernels as the call, without the launch
        gaps between them."""
        torch = self.torch
        self.graphs = {}
        for name, fn in self.parts():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            self.graphs[name] = g
        torch.cuda.synchronize()

    def step(self, marks=None):
        """The whole path; ``marks`` (dict of event pairs) brackets the parts."""
        graphs = getattr(self, "graphs", None)
        for name, fn in self.parts():
            if marks:
                marks[name][0].record()
            if graphs:
                graphs[name].replay()
            else:
                fn()
            if marks:
                marks[name][1].record()


def run_gpu(args, rank, world, local_rank):
    import torch
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    prob = make_problem(args)
    st = GpuStep(prob, torch, rx, args.extend_path, args.rope, getattr(args, "kv_fp8", False))
    flush = L2Flush(torch)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush()
        st.step()
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise RuntimeError(f"device status {int(st.status.item())} after warm-up")
    if args.graph:
        st.capture()
        for _ in range(args.warmup):
            flush()
            st.step()
        torch.cuda.synchronize()

    E = torch.cuda.Event
    parts = [name for name, _ in st.parts()]
    marks = [{k: (E(enable_timing=True), E(enable_timing=True)) for k in parts}
             for _ in range(args.steps)]
    steps_ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()
            steps_ev[i][0].record()
            st.step(marks[i])
            steps_ev[i][1].record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    if int(st.status.item()) != 0:
        raise RuntimeError(f"device status {int(st.status.item())} after the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in steps_ev]
    part_ms = {k: [m[k][0].elapsed_time(m[k][1]) for m in marks] for k in parts}
    tot_ms = max_over_ranks(sum(step_ms), dist, "cuda")
    ms_per_step = tot_ms / args.steps

    # end to end through the public API: pinned host inputs in, result out
    if dist:
        dist.barrier()
    e2e = run_e2e(st, torch, rx, args.steps, flush, dist, world)
    if int(st.status.item()) != 0:
        raise RuntimeError(f"device status {int(st.status.item())} after the end-to-end steps")

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    hbm, tflops, tflops_sus, peak_src = measured_peaks()
    B_dec = len(prob.dec_req_idx)
    flops_ext = prob.extend_flops()
    kv_row = prob.kv_row_bytes
    out = {}
    if st.has_dec:
        value = job_throughput(B_dec, world, args.steps, tot_ms)
        metric, unit = "decode tok/s", "tok/s"
        dec_ms = statistics.mean(part_ms["decode"])
        uniq_bytes = st.plan_info.tokens_read * kv_row
        achieved = uniq_bytes / (dec_ms / 1e3) / 1e9
        traffic, tsrc = profiled_traffic(args.workload, "decode")
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic, "traffic_source": tsrc,
                "kernel": "rx_attn_decode (" + " + ".join(st.decode_kernels) + ")",
                "algorithmic_bytes_per_launch": int(uniq_bytes), "launch_ms": round(dec_ms, 5),
                "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)",
                "frac_of_8000": round(achieved / 8000.0, 4)}
        out["decode"] = {"tok_s": B_dec / (dec_ms / 1e3), "hbm_gbs_unique": achieved,
                         "unique_kv_bytes": int(uniq_bytes),
                         "dense_kv_bytes": int(prob.decode_dense_tokens() * kv_row),
                         "ms": dec_ms, "segments": st.plan_info.n_segments,
                         "work_items": st.plan_info.n_items, "kv_chunk": st.plan_info.kv_chunk}
    if st.has_ext:
        ext_ms = statistics.mean(part_ms["extend"])
        tf = flops_ext / (ext_ms / 1e3) / 1e12
        out["extend"] = {"tflops": tf, "ms": ext_ms, "tok_s": float(np.sum(prob.ext_extend_len)) / (ext_ms / 1e3),
                         "flops": int(flops_ext), "frac_of_burst": tf / tflops}
        if not st.has_dec:
            metric, unit = "extend TFLOPS", "TFLOP/s"
            value = job_throughput(flops_ext, world, args.steps, tot_ms) / 1e12
            traffic, tsrc = profiled_traffic(args.workload, args.extend_path)
            roof = {"bound": "tensor", "achieved": round(tf, 2), "peak": tflops, "unit": "TFLOP/s",
                    "frac": round(tf / tflops, 4), "traffic": traffic, "traffic_source": tsrc,
                    "kernel": "rx_attn_extend (" + ("offsets + staging copy + extend_kernel"
                                                    if args.extend_path == "staged" else "extend_kernel") + ")",
                    "algorithmic_flops_per_launch": int(flops_ext), "launch_ms": round(ext_ms, 5),
                    "peak_source": f"{peak_src} bf16_tflops (burst)"}
    out["kv_store"] = {"ms": statistics.mean(part_ms["store"]),
                       "gbs": 2 * len(prob.new_slots) * kv_row / (statistics.mean(part_ms["store"]) / 1e3) / 1e9}
    if st.kv_fp8:
        f8 = statistics.mean(part_ms["store_fp8"])
        n_vals = len(prob.new_slots) * prob.hkv * prob.d
        out["kv_store_fp8"] = {"ms": f8, "gbs": 2 * n_vals * (2 + 1) / (f8 / 1e3) / 1e9}
    if st.rope_base:
        # K rotated inside the store (above); q rows rotated in place: read and
        # write of every q row
        q_bytes = 2 * (prob.q_ext.size + prob.q_dec.size) * 2
        rq = statistics.mean(part_ms["rope_q"])
        out["kv_store"]["rope_base"] = st.rope_base
        out["rope_q"] = {"ms": rq, "gbs": q_bytes / (rq / 1e3) / 1e9}
    line = {
        "metric": f"prefix-shared attn: {metric}", "value": round(value, 3), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random slot permutation)",
        "config": workload_config(prob, args.workload, world, args.extend_path, getattr(args, "graph", False),
                                  getattr(args, "rope", 0.0)),
        "roofline": roof, "e2e": e2e, "gpu_launches": st.launches * args.steps,
        "clocks": clk.summary(), "parts": out, "wall_s_timed_loop": round(t_wall, 3),
    }
    if st.kv_fp8:
        line["config"]["kv_fp8"] = "extra part: the step's K/V rows also stored as E4M3 codes (scale 1)"
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob, args.workload, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of every rank's value: the slowest replica sets the job's
    time.  A collective, so every rank calls it; `dist` None means one rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class L2Flush:
    """Run between timed steps: writes a buffer twice the size of L2 (no input
    of the step stays cached), then reads another one of the same size, which
    evicts the dirty lines of the write (the step would otherwise pay for
    writing them back) and leaves L2 holding clean lines of no use to it."""

    def __init__(self, torch):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 2, dtype=torch.bfloat16, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.acc = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.acc)


def job_throughput(units_per_rank_step: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's
    time (weak scaling: each rank carries the full per-GPU workload)."""
    return units_per_rank_step * world * steps / (max_ms / 1e3)


def run_e2e(st, torch, rx, steps, flush, dist=None, world=1):
    """Per step: pinned host -> device copies of the step's inputs, the path,
    device -> host copy of its outputs; timed with events on the stream."""
    p = st.prob
    s = torch.cuda.current_stream()
    h_in = [st.k_new.cpu().pin_memory(), st.v_new.cpu().pin_memory(), st.slots.cpu().pin_memory()]
    d_in = [st.k_new, st.v_new, st.slots]
    outs = []
    if st.has_ext:
        h_in.append(st.q_ext.cpu().pin_memory())
        d_in.append(st.q_ext)
        outs.append(st.o_ext)
    if st.has_dec:
        h_in.append(st.q_dec.cpu().pin_memory())
        d_in.append(st.q_dec)
        outs.append(st.o_dec)
    h_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    n = max(3, min(steps, 200))
    E = torch.cuda.Event
    ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        ev[i][0].record()
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        st.step()
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / n, dist, "cuda")
    h2d = sum(h.numel() * h.element_size() for h in h_in)
    d2h = sum(h.numel() * h.element_size() for h in h_out)
    if st.has_dec:
        val, unit = job_throughput(len(p.dec_req_idx), world, 1, ms), "tok/s"
    else:
        val, unit = job_throughput(p.extend_flops(), world, 1, ms) / 1e12, "TFLOP/s"
    return {"value": round(val, 3), "unit": unit, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 5), "steps": n}


# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# captures summarised in the named profile; an entry is removed whenever its
# kernel changes, so that an old count is never reported for new code.
PROFILED_TRAFFIC = {
    ("few_shot_decode", "decode"): (298_800_000, "profiles/decode_kernel.few_shot_decode.md"),
    ("tree_of_thought_decode", "decode"): (401_500_000, "profiles/decode_gqa_kernel.tree_of_thought_decode.md"),
    ("cached_prefix_extend", "staged"): (585_800_000, "profiles/extend_kernel.cached_prefix_extend.md"),
    ("constrained_decode", "fsm"): (132_300_000, "profiles/fsm_scan_kernel.constrained_decode.md"),
}


def profiled_traffic(workload, part):
    hit = PROFILED_TRAFFIC.get((workload, part))
    return (hit[0], hit[1]) if hit else (None, None)


TREE_WORKLOADS = ("mixed_chat",)
WORKLOADS = sorted(list(inputs.FULL_SIZE) + list(TREE_WORKLOADS))


def make_problem(args, admit_with="library"):
    """The workload's batch.  The long multi-turn chat batch is admitted into
    its full pool through a radix cache: the library's (``admit_with`` =
    "library") or, for the reference arm, the oracle's trie ("oracle"); both
    hand out the same slot lists (a CPU test checks it bit for bit)."""
    kw = {}
    if args.pool_slots:
        kw["num_slots"] = args.pool_slots
    if args.workload not in TREE_WORKLOADS:
        return inputs.FULL_SIZE[args.workload](**kw)
    scn = inputs.mixed_chat_scenario(**kw)
    if admit_with == "oracle":
        from oracle import tree_ref
        _, out = tree_ref.replay(scn.free_order, scn.prefill, scn.batch)
        rows, ks = [np.asarray(r, np.int32) for r, _, _ in out], [k for _, k, _ in out]
    else:
        from prefix_shared_kv_radixattention_gb300 import admission
        adm = admission.replay(scn)
        rows, ks = adm.rows, adm.prefix_lens
    return inputs.problem_from_admission(scn, rows, ks)


def workload_config(prob, name, world, extend_path="staged", graph=False, rope=0.0):
    cfg = {"workload": name, "hq": prob.hq, "hkv": prob.hkv, "head_dim": prob.d,
           "pool_slots": prob.num_slots, "decode_requests": int(len(prob.dec_req_idx)),
           "extend_requests": int(len(prob.ext_req_idx)),
           "l2": "between timed steps: 256 MiB written (evicts the step's inputs), then 256 MiB read "
                 "(evicts the write's dirty lines)",
           "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
           "launch": "CUDA graph per part" if graph else "direct calls"}
    if len(prob.dec_req_idx):
        cfg["decode_context"] = int(prob.dec_seq_len.max())
    if len(prob.ext_req_idx):
        cfg["extend_prefix"] = int(prob.ext_prefix_len.max())
        cfg["extend_new"] = int(prob.ext_extend_len.max())
        cfg["extend_path"] = extend_path
    if rope:
        cfg["rope_base"] = rope
    return cfg


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------


def _oracle_pools(prob):
    import oracle
    slots = np.concatenate([prob.cached_slots, prob.new_slots])
    uniq = np.unique(slots)
    kp = np.zeros((len(uniq), prob.hkv, prob.d), np.uint16)
    vp = np.zeros_like(kp)
    pos = np.searchsorted(uniq, prob.cached_slots)
    kp[pos], vp[pos] = prob.cached_k, prob.cached_v
    oracle.kv_store(kp, vp, prob.new_k, prob.new_v, np.searchsorted(uniq, prob.new_slots).astype(np.int32))
    rtt = prob.req_to_token
    loc = np.minimum(np.searchsorted(uniq, np.maximum(rtt, 0)), len(uniq) - 1)
    rtt_c = np.where((rtt >= 0) & (uniq[loc] == rtt), loc, -1).astype(np.int32)
    return kp, vp, rtt_c


def oracle_sample(prob, pools, rows_dec, rows_ext_tokens, threads):
    """One bounded oracle pass: the first rows_dec decode rows and the last
    rows_ext_tokens extend tokens of each extend request.  Returns
    (seconds, decode rows done, extend flops done)."""
    import oracle
    kp, vp, rtt = pools
    flops = 0
    nd = 0
    t0 = time.perf_counter()
    if len(prob.dec_req_idx) and rows_dec:
        nd = min(rows_dec, len(prob.dec_req_idx))
        oracle.decode(prob.q_dec[:nd], kp, vp, rtt, prob.dec_req_idx[:nd], prob.dec_seq_len[:nd],
                      prob.sm_scale, n_threads=threads)
    if len(prob.ext_req_idx) and rows_ext_tokens:
        q_rows, kend, qi = [], [], []
        for b in range(len(prob.ext_req_idx)):
            E, P = int(prob.ext_extend_len[b]), int(prob.ext_prefix_len[b])
            for i in range(max(0, E - rows_ext_tokens), E):
                qi.append(int(prob.qo_indptr[b]) + i)
                q_rows.append(int(prob.ext_req_idx[b]))
                kend.append(P + i + 1)
        kend = np.array(kend, np.int32)
        oracle.attention(prob.q_ext[qi], kp, vp, rtt, np.array(q_rows, np.int32), np.zeros_like(kend),
                         kend, prob.sm_scale, n_threads=threads)
        flops = int(4 * prob.d * prob.hq * kend.astype(np.int64).sum())
    return time.perf_counter() - t0, nd, flops


def cpu_baseline(prob, name, budget_s=15.0):
    """The oracle as it stands, on all host cores, repeated over a bounded
    sample until about budget_s seconds of CPU work are done."""
    threads = cores()
    pools = _oracle_pools(prob)
    has_dec = len(prob.dec_req_idx) > 0
    tot, work, reps = 0.0, 0, 0
    if has_dec:
        rows = len(prob.dec_req_idx)
        sec, _, _ = oracle_sample(prob, pools, 1, 0, threads)
        rows = int(max(1, min(rows, budget_s / max(sec, 1e-4))))
        while tot < budget_s and reps < 10000:
            sec, nd, _ = oracle_sample(prob, pools, rows, 0, threads)
            tot, work, reps = tot + sec, work + nd, reps + 1
        return {"value": round(work / tot, 3), "unit": "tok/s", "cores": threads, "kind": "oracle",
                "sample": f"{rows} of {len(prob.dec_req_idx)} decode rows of {name} (all heads, fp64), "
                          f"repeated {reps} times", "seconds": round(tot, 3)}
    sec, _, _ = oracle_sample(prob, pools, 0, 1, threads)
    toks = int(max(1, min(int(prob.ext_extend_len.min()), budget_s / max(sec, 1e-4))))
    while tot < budget_s and reps < 10000:
        sec, _, fl = oracle_sample(prob, pools, 0, toks, threads)
        tot, work, reps = tot + sec, work + fl, reps + 1
    return {"value": round(work / tot / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"last {toks} extend tokens of each of {len(prob.ext_req_idx)} requests of {name} "
                      f"(fp64), repeated {reps} times", "seconds": round(tot, 3)}


# ---------------------------------------------------------------------------
# constrained decoding (compressed finite-state machine)
# ---------------------------------------------------------------------------

FSM_WORKLOAD = "constrained_decode"
FSM_SHAPE = {"vocab": 128256, "batch": 256, "n_fields": 8, "max_jump": 16}


def fsm_problem():
    from prefix_shared_kv_radixattention_gb300 import fsm_inputs
    a = fsm_inputs.json_automaton(vocab=FSM_SHAPE["vocab"], n_fields=FSM_SHAPE["n_fields"])
    state, logits = fsm_inputs.step_inputs(a, FSM_SHAPE["batch"])
    return a, state, logits


def fsm_config(a, world):
    return {"workload": FSM_WORKLOAD, "vocab": a.vocab, "batch": FSM_SHAPE["batch"], "states": a.n_states,
            "edges": int(len(a.tok)), "max_jump": FSM_SHAPE["max_jump"], "constraint": a.schema_text,
            "l2": "between timed steps: 256 MiB written (evicts the step's inputs), then 256 MiB read "
                  "(evicts the write's dirty lines)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "launch": "direct calls"}


def fsm_oracle_sample(a, jumps, ends, state, logits, n):
    """The oracle's step over the first n requests; (seconds, requests)."""
    from oracle import fsm as ofsm
    t0 = time.perf_counter()
    ofsm.step(logits[:n], state[:n], a.row_ptr, a.tok, a.nxt, jumps, ends)
    return time.perf_counter() - t0, n


def run_gpu_fsm(args, rank, world, local_rank):
    import torch
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    a, state0, logits = fsm_problem()
    B, V, J = FSM_SHAPE["batch"], a.vocab, FSM_SHAPE["max_jump"]
    m = rx.Fsm(a.n_states, a.vocab, a.row_ptr, a.tok, a.nxt, J)
    lg = torch.from_numpy(logits).cuda()
    st0 = torch.from_numpy(state0).cuda()
    st = st0.clone()
    out = torch.zeros((B, 1 + J), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = rx.fsm_workspace(B)
    flush = L2Flush(torch)
    E = torch.cuda.Event

    def step(marks=None):
        st.copy_(st0)                   # every step starts from the batch's states
        if marks:
            marks[0].record()
        rx.rx_fsm_step(m, lg, st, out, cnt, ws, status)
        if marks:
            marks[1].record()

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")
    marks = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(args.steps)]
    steps_ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()
            steps_ev[i][0].record()
            step(marks[i])
            steps_ev[i][1].record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed steps")
    tot_ms = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in steps_ev), dist, "cuda")
    k_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in marks)
    emitted = cnt.cpu().numpy()
    # end to end: pinned host logits and states in, tokens and counts out
    h_lg = torch.from_numpy(logits).pin_memory()
    h_st = torch.from_numpy(state0).pin_memory()
    h_out = torch.empty((B, 1 + J), dtype=torch.int32, pin_memory=True)
    h_cnt = torch.empty(B, dtype=torch.int32, pin_memory=True)
    n = max(3, min(args.steps, 200))
    ev = [(E(enable_timing=True), E(enable_timing=True)) for _ in range(n)]
    if dist:
        dist.barrier()
    for i in range(n):
        flush()
        ev[i][0].record()
        lg.copy_(h_lg, non_blocking=True)
        st.copy_(h_st, non_blocking=True)
        rx.rx_fsm_step(m, lg, st, out, cnt, ws, status)
        h_out.copy_(out, non_blocking=True)
        h_cnt.copy_(cnt, non_blocking=True)
        ev[i][1].record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in ev), dist, "cuda")
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the end-to-end steps")
    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    hbm, _, _, peak_src = measured_peaks()
    W = (V + 31) // 32
    algo = B * (V * 4 + W * 4)          # each request's logits row and its state's mask row
    achieved = algo / (k_ms / 1e3) / 1e9
    traffic, tsrc = profiled_traffic(FSM_WORKLOAD, "fsm")
    line = {
        "metric": "constrained decode: requests/s", "value": round(job_throughput(B, world, args.steps, tot_ms), 3),
        "unit": "req/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded JSON-object constraint, N(0,1) fp32 logits)",
        "config": fsm_config(a, world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic, "traffic_source": tsrc,
                     "kernel": "rx_fsm_step (fsm_scan_kernel + fsm_finish_kernel)",
                     "algorithmic_bytes_per_launch": int(algo),
                     "launch_ms": round(k_ms, 5), "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"},
        "e2e": {"value": round(job_throughput(B, world, n, e2e_ms), 3), "unit": "req/s",
                "h2d_bytes_per_step": int(logits.nbytes + state0.nbytes),
                "d2h_bytes_per_step": int(out.numel() * 4 + cnt.numel() * 4), "ms_per_step": round(e2e_ms / n, 5),
                "steps": n},
        "gpu_launches": 2 * args.steps, "clocks": clk.summary(),
        "parts": {"fsm_step": {"ms": k_ms, "tokens_per_step": float(emitted.mean()),
                               "jump_tokens_per_step": float(emitted.mean() - 1.0)}},
        "wall_s_timed_loop": round(t_wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        from oracle import fsm as ofsm
        jumps, ends, _ = ofsm.compress(a.n_states, a.row_ptr, a.tok, a.nxt, J)
        tot, work, reps = 0.0, 0, 0
        while tot < args.cpu_seconds and reps < 1000:
            sec, nr = fsm_oracle_sample(a, jumps, ends, state0, logits, B)
            tot, work, reps = tot + sec, work + nr, reps + 1
        line["cpu_baseline"] = {"value": round(work / tot, 3), "unit": "req/s", "cores": 1, "kind": "oracle",
                                "sample": f"the oracle's step over all {B} requests, repeated {reps} times",
                                "seconds": round(tot, 3)}
    print(json.dumps(line), flush=True)


def run_reference_fsm(args, rank, world):
    if rank != 0:
        return
    from oracle import fsm as ofsm
    a, state0, logits = fsm_problem()
    B, J = FSM_SHAPE["batch"], FSM_SHAPE["max_jump"]
    jumps, ends, _ = ofsm.compress(a.n_states, a.row_ptr, a.tok, a.nxt, J)
    secs = []
    for i in range(args.warmup + args.steps):
        s, _ = fsm_oracle_sample(a, jumps, ends, state0, logits, B)
        if i >= args.warmup:
            secs.append(s)
    tot = sum(secs)
    value = B * args.steps / tot
    line = {"impl": "reference", "metric": "constrained decode: requests/s", "value": round(value, 3),
            "unit": "req/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (argmax), int", "data": "synthetic (seeded JSON-object constraint)",
            "config": fsm_config(a, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "req/s", "cores": 1, "kind": "oracle",
                             "sample": f"the oracle's step over all {B} requests per step"},
            "e2e": {"value": round(value, 3), "unit": "req/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    prob = make_problem(args, admit_with="oracle")
    threads = cores()
    pools = _oracle_pools(prob)
    has_dec = len(prob.dec_req_idx) > 0
    # a step = a bounded sample of the workload, sized to a few seconds
    sec1, _, _ = oracle_sample(prob, pools, 1 if has_dec else 0, 0 if has_dec else 1, threads)
    budget = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    n = int(max(1, budget / max(sec1, 1e-4)))
    secs, work = [], []
    for i in range(args.warmup + args.steps):
        if has_dec:
            s, nd, _ = oracle_sample(prob, pools, min(n, len(prob.dec_req_idx)), 0, threads)
            w = nd
        else:
            s, _, fl = oracle_sample(prob, pools, 0, min(n, int(prob.ext_extend_len.min())), threads)
            w = fl
        if i >= args.warmup:
            secs.append(s)
            work.append(w)
    tot = sum(secs)
    if has_dec:
        value, unit, metric = sum(work) / tot, "tok/s", "decode tok/s"
        sample = f"{work[0]} of {len(prob.dec_req_idx)} decode rows per step, all heads, fp64"
    else:
        value, unit, metric = sum(work) / tot / 1e12, "TFLOP/s", "extend TFLOPS"
        sample = f"last {min(n, int(prob.ext_extend_len.min()))} extend tokens per request per step, fp64"
    line = {"impl": "reference", "metric": f"prefix-shared attn: {metric}", "value": round(value, 6),
            "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16, random slot permutation)",
            "config": workload_config(prob, args.workload, world, args.extend_path, getattr(args, "graph", False),
                                  getattr(args, "rope", 0.0)),
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="few_shot_decode", choices=WORKLOADS + [FSM_WORKLOAD])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool-slots", type=int, default=0,
                    help="override the pool size (profiling runs on a smaller device footprint)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="also store the step's K/V rows into FP8 (E4M3) pools (an extra part of the step)")
    ap.add_argument("--rope", type=float, default=0.0, metavar="BASE",
                    help="add rotary position embedding to the step (K fused into the store, q in place)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each part of the timed step as a CUDA graph of the same calls")
    ap.add_argument("--extend-path", default="staged", choices=["staged", "gather"],
                    help="extend through a staging workspace (default) or gathering rows in the attention kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.workload == FSM_WORKLOAD:
        if args.impl == "reference":
            run_reference_fsm(args, rank, world)
        else:
            run_gpu_fsm(args, rank, world, local_rank)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
