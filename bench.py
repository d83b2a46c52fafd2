"""Benchmark of the prefix-shared KV attention path on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole path over one batch of synthetic input: the
KV store of the step's new tokens, then the attention the workload needs
(decode with its decode plan, and/or extend).  Inputs are resident in HBM
before timing starts; between timed steps a 256 MiB buffer is written, so that
no KV survives in L2 (129 MB), and a second 256 MiB buffer is read, so that the
lines the write left dirty are written back before the step rather than
inside it; each step is timed with CUDA events on the launching stream.  The
decode plan is built once per batch, before timing, from the host copy of
req_to_token (its time is reported); it stays valid for the batch's later
decode steps, since each request's last piece follows its length on the
device.

Workloads (default: mixed_chat, the largest configuration that fits one GPU):
  mixed_chat              16 decode x 32k + 16 extend x (4096 + 1024), 64/8,
                          admitted through the radix cache into a full
                          1M-slot pool (LRU eviction of cold conversations)
  few_shot_decode         64 x (1024 shared + 256 private + 1), MHA 32x128, 2M slots
  tree_of_thought_decode  256 leaves of a depth-4 fanout-4 tree, GQA 32/8
  cached_prefix_extend    32 x (2048 cached + 512 new), GQA 32/8
  tiny_extend             4 x (64 cached + 16 new), 4 heads, head_dim 64
  constrained_decode      one compressed-FSM decoding step (masked argmax and
                          jump) for 256 requests over a 128,256-id vocabulary
                          under a JSON-object constraint

One JSON line is printed by rank 0: "roofline" describes the step's dominant
part (the longer of extend and decode), "rooflines" every part.  "e2e" runs
the same step through the public API one synchronized step at a time, with
the step's inputs copied in from pinned host memory and its outputs copied
back.  Under torchrun every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); value = work of all
ranks / the slowest rank's time.

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
            t0 = time.perf_counter()
            buf, info = rx.rx_decode_plan_build(p.req_to_token, p.dec_req_idx, p.dec_seq_len, p.hq, p.hkv)
            self.plan_build_ms = (time.perf_counter() - t0) * 1e3
            self.plan_info = info
            self.plan = rx.plan_to_device(buf, info, B)
            # bytes the call moves besides the unique K/V rows: q read, o
            # written, the plan and slot ids read, and the fp32 partials
            # (o and log2-sum-exp) of split rows, written once and read back
            nparts = np.asarray(buf[B:2 * B], np.int64)
            split = nparts[nparts > 1]
            self.overhead_bytes = {
                "q": int(B * p.hq * p.d * 2), "o": int(B * p.hq * p.d * 2),
                "plan_and_slot_ids": int(len(buf) * 4 + info.tokens_read * 4),
                "partials": int(2 * split.sum() * p.hq * (p.d + 1) * 4)}
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
                self.launches += 3  # shared-tile search + packed-row offsets + row copy
        # FP8 pools (optional): the whole step on E4M3 pools
        self.kv_fp8 = kv_fp8
        if kv_fp8:
            # E4M3 pools (scale 1): the cached rows quantized at set-up, the
            # step's rows stored by rx_kv_store_fp8 in the timed step (in place
            # of the bf16 store); extend and decode read them
            # (rx_attn_extend_fp8, rx_attn_decode_fp8)
            self.k8 = torch.zeros((p.num_slots, p.hkv, p.d), dtype=torch.uint8, device=dev)
            self.v8 = torch.zeros_like(self.k8)
            for s0 in range(0, len(idx), 1 << 16):
                sl = idx[s0:s0 + (1 << 16)].to(torch.int32)
                rx.rx_kv_store_fp8(self.k8, self.v8, 1.0, 1.0, self.k_pool[sl.long()], self.v_pool[sl.long()], sl,
                                   self.status)
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
        if self.kv_fp8:
            self.rx.rx_attn_decode_fp8(self.k8, self.v8, 1.0, 1.0, self.q_dec, self.o_dec, None, self.dec_req,
                                       self.dec_len, self.rtt, self.max_len, p.sm_scale, self.plan, self.ws,
                                       self.status)
            return
        self.rx.rx_attn_decode(self.k_pool, self.v_pool, self.q_dec, self.o_dec, None, self.dec_req,
                               self.dec_len, self.rtt, self.max_len, p.sm_scale, self.plan, self.ws,
                               self.status)

    def extend(self):
        p = self.prob
        if self.kv_fp8:
            self.rx.rx_attn_extend_fp8(self.k8, self.v8, 1.0, 1.0, self.q_ext, self.o_ext, None, self.qo,
                                       self.ext_req, self.ext_P, self.ext_E, self.rtt, self.max_E, p.sm_scale,
                                       self.ext_ws, self.status)
            return
        self.rx.rx_attn_extend(self.k_pool, self.v_pool, self.q_ext, self.o_ext, None, self.qo,
                               self.ext_req, self.ext_P, self.ext_E, self.rtt, self.max_E, p.sm_scale,
                               self.status, workspace=self.ext_ws)

    def store_fp8(self):
        if self.rope_base:
            self.rx.rx_kv_store_rope_fp8(self.k8, self.v8, 1.0, 1.0, self.k_new, self.v_new, self.slots,
                                         self.pos_new, self.rope_base, self.status)
        else:
            self.rx.rx_kv_store_fp8(self.k8, self.v8, 1.0, 1.0, self.k_new, self.v_new, self.slots, self.status)

    def parts(self):
        return ([("store_fp8", self.store_fp8)] if self.kv_fp8 else [("store", self.kv_store)]) + \
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
    out, roofs = {}, {}
    ms_of = {k: statistics.mean(v) for k, v in part_ms.items()}
    if st.has_dec:
        dec_ms = ms_of["decode"]
        uniq_bytes = st.plan_info.tokens_read * (kv_row // 2 if st.kv_fp8 else kv_row)
        achieved = uniq_bytes / (dec_ms / 1e3) / 1e9
        traffic, tsrc = profiled_traffic(args.workload, "decode_fp8" if st.kv_fp8 else "decode")
        roofs["decode"] = {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": traffic, "traffic_source": tsrc,
            "kernel": ("rx_attn_decode_fp8 (" + " + ".join(k if k == "merge_kernel" else k + "<F8>"
                                                           for k in st.decode_kernels) + ")" if st.kv_fp8 else
                       "rx_attn_decode (" + " + ".join(st.decode_kernels) + ")"),
            "algorithmic_bytes_per_launch": int(uniq_bytes), "launch_ms": round(dec_ms, 5),
            "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)", "frac_of_8000": round(achieved / 8000.0, 4)}
        out["decode"] = {"tok_s": B_dec / (dec_ms / 1e3), "hbm_gbs_unique": achieved,
                         "unique_kv_bytes": int(uniq_bytes),
                         "dense_kv_bytes": int(prob.decode_dense_tokens() * kv_row),
                         "ms": dec_ms, "segments": st.plan_info.n_segments,
                         "work_items": st.plan_info.n_items, "kv_chunk": st.plan_info.kv_chunk,
                         "plan_build_ms_once_per_batch": round(st.plan_build_ms, 3),
                         "overhead_bytes": st.overhead_bytes}
    if st.has_ext:
        ext_ms = ms_of["extend"]
        tf = flops_ext / (ext_ms / 1e3) / 1e12
        traffic, tsrc = profiled_traffic(args.workload, args.extend_path + ("_fp8" if st.kv_fp8 else ""))
        roofs["extend"] = {
            "bound": "tensor", "achieved": round(tf, 2), "peak": tflops, "unit": "TFLOP/s",
            "frac": round(tf / tflops, 4), "traffic": traffic, "traffic_source": tsrc,
            "kernel": ("rx_attn_extend_fp8" if st.kv_fp8 else "rx_attn_extend") + " (" +
                      ("shared-tile search + offsets + staging copy + extend_kernel"
                       if args.extend_path == "staged" else "extend_kernel") + ")",
            "algorithmic_flops_per_launch": int(flops_ext), "launch_ms": round(ext_ms, 5),
            "peak_source": f"{peak_src} bf16_tflops (burst)",
            "frac_of_sustained": round(tf / tflops_sus, 4) if tflops_sus else None}
        out["extend"] = {"tflops": tf, "ms": ext_ms, "tok_s": float(np.sum(prob.ext_extend_len)) / (ext_ms / 1e3),
                         "flops": int(flops_ext), "frac_of_burst": tf / tflops}
    metric, unit, per_step = step_metric(prob)
    value = job_throughput(per_step, world, args.steps, tot_ms)
    # the dominant part of the step (the longer of extend and decode) is the
    # kernel the line's roofline describes; both are in "rooflines"
    dominant = max(roofs, key=lambda k: roofs[k]["launch_ms"])
    if not st.kv_fp8:
        out["kv_store"] = {"ms": ms_of["store"],
                           "gbs": 2 * len(prob.new_slots) * kv_row / (ms_of["store"] / 1e3) / 1e9}
    else:
        f8 = ms_of["store_fp8"]
        n_vals = len(prob.new_slots) * prob.hkv * prob.d
        out["kv_store_fp8"] = {"ms": f8, "gbs": 2 * n_vals * (2 + 1) / (f8 / 1e3) / 1e9}
    if st.rope_base:
        # K rotated inside the store (above); q rows rotated in place: read and
        # write of every q row
        q_bytes = 2 * (prob.q_ext.size + prob.q_dec.size) * 2
        rq = ms_of["rope_q"]
        out["kv_store_fp8" if st.kv_fp8 else "kv_store"]["rope_base"] = st.rope_base
        out["rope_q"] = {"ms": rq, "gbs": q_bytes / (rq / 1e3) / 1e9}
    line = {
        "metric": f"prefix-shared attn: {metric}", "value": round(value, 3), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random slot permutation)",
        "config": workload_config(prob, args.workload, world, args.extend_path, getattr(args, "graph", False),
                                  getattr(args, "rope", 0.0)),
        "roofline": dict(roofs[dominant], part=dominant), "rooflines": roofs, "e2e": e2e,
        "gpu_launches": st.launches * args.steps,
        "clocks": clk.summary(), "parts": out, "wall_s_timed_loop": round(t_wall, 3),
    }
    if st.kv_fp8:
        line["config"]["kv_fp8"] = ("the step on E4M3 pools (scale 1; cached rows quantized at set-up): its K/V "
                                    "rows stored as codes, extend and decode over the codes")
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob, args.workload, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def step_metric(prob):
    """(metric, unit, units per step) of a workload's step: decode tokens
    for decode batches, TFLOP for extend batches, and for a mixed batch the
    tokens it carries (one per decode request plus every extend token)."""
    n_dec, n_ext = len(prob.dec_req_idx), int(np.sum(prob.ext_extend_len))
    if n_dec and n_ext:
        return "tok/s (decode + extend tokens of the mixed step)", "tok/s", float(n_dec + n_ext)
    if n_dec:
        return "decode tok/s", "tok/s", float(n_dec)
    return "extend TFLOPS", "TFLOP/s", prob.extend_flops() / 1e12


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


class E2EPipeline:
    """One step of the path as a caller drives it through the public API with
    host buffers, its copies overlapped with the kernels.  An input stream
    brings in, in this order: the decode requests' new K/V rows, slots and
    queries; then, per chunk of extend requests, the chunk's new K/V rows,
    slots and queries.  The compute stream stores the decode rows as soon as
    they are in (while the queries arrive) and runs decode once its queries
    are in too; each chunk's rows are stored as soon as they are in, and its
    extend run (rx_attn_extend over the chunk) once its queries are in, the
    chunks alternating between two compute streams with a staging workspace
    each (different chunks touch disjoint rows and slots, so one chunk's
    staging and last wave overlap the next one's attention); an output
    stream copies each result back as soon as it is written.  The host link
    (about 200 GB/s each way on this machine) is slower than the kernels,
    so decode goes first (its inputs are small,
    and it runs while the first chunk arrives) and the chunks grow, then
    shrink (little to wait for at the start, little to copy back after the
    last kernel).  Where a chunk's new rows are not one contiguous range of
    the step's rows, every new row goes in before the first store instead.
    The same calls, on the same data, as the step."""

    FRACTIONS = (0.12, 0.2, 0.24, 0.2, 0.14, 0.1)   # extend requests per chunk, in order

    def __init__(self, st, torch, rx, fractions=FRACTIONS):
        self.st, self.torch, self.rx = st, torch, rx
        p = st.prob
        pin = lambda t: t.cpu().pin_memory()
        self.h_k, self.h_v, self.h_sl = pin(st.k_new), pin(st.v_new), pin(st.slots)
        self.h_in, self.h_out = [self.h_k, self.h_v, self.h_sl], []
        # with RoPE the positions are inputs of the step too: of the new
        # rows, of the decode queries and of the extend queries
        self.h_pos = {}
        if st.rope_base:
            self.h_pos["new"] = pin(st.pos_new)
            if st.has_dec:
                self.h_pos["dec"] = pin(st.pos_dec)
            if st.has_ext:
                self.h_pos["ext"] = pin(st.pos_ext)
            self.h_in += list(self.h_pos.values())
        # the new row of each slot: which rows the decode part and each chunk store
        row_of = {int(s): i for i, s in enumerate(p.new_slots)}
        n_new = len(p.new_slots)

        def rows_of(slots):
            idx = sorted(row_of[int(s)] for s in slots if int(s) in row_of)
            return (idx[0], idx[-1] + 1) if idx and idx[-1] - idx[0] + 1 == len(idx) else None

        covered = 0
        self.dec_rows = (0, 0)
        if st.has_dec:
            self.h_qd = [pin(st.q_dec), pin(st.dec_len)]
            self.h_od = torch.empty(st.o_dec.shape, dtype=st.o_dec.dtype, pin_memory=True)
            self.h_in += self.h_qd
            self.h_out.append(self.h_od)
            dec_slots = [p.req_to_token[r, L - 1] for r, L in zip(p.dec_req_idx, p.dec_seq_len)]
            self.dec_rows = rows_of(dec_slots) or (0, 0)
            covered += self.dec_rows[1] - self.dec_rows[0]
        self.chunks = []
        if st.has_ext:
            self.h_qe = pin(st.q_ext)
            self.h_oe = torch.empty(st.o_ext.shape, dtype=st.o_ext.dtype, pin_memory=True)
            self.h_in.append(self.h_qe)
            self.h_out.append(self.h_oe)
            Be = len(p.ext_req_idx)
            n = min(len(fractions), Be)
            fr = np.asarray(fractions[:n], np.float64)
            cuts = np.round(np.cumsum(np.concatenate([[0.0], fr / fr.sum()])) * Be).astype(int)
            cuts = sorted(set(int(x) for x in cuts))
            i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
            max_ctx, max_n = 0, 0
            for b0, b1 in zip(cuts[:-1], cuts[1:]):
                r0, r1 = int(p.qo_indptr[b0]), int(p.qo_indptr[b1])
                ctx = int((p.ext_prefix_len[b0:b1] + p.ext_extend_len[b0:b1]).sum())
                max_ctx, max_n = max(max_ctx, ctx), max(max_n, b1 - b0)
                new_slots = np.concatenate([p.req_to_token[r, P:P + E] for r, P, E in
                                            zip(p.ext_req_idx[b0:b1], p.ext_prefix_len[b0:b1],
                                                p.ext_extend_len[b0:b1])])
                kv = rows_of(new_slots) or (0, 0)
                covered += kv[1] - kv[0]
                self.chunks.append(dict(
                    rows=(r0, r1), kv=kv, qo=i32(p.qo_indptr[b0:b1 + 1] - r0), req=i32(p.ext_req_idx[b0:b1]),
                    P=i32(p.ext_prefix_len[b0:b1]), E=i32(p.ext_extend_len[b0:b1]),
                    max_E=int(p.ext_extend_len[b0:b1].max()), n=b1 - b0))
            # one staging workspace per compute stream (the chunks alternate)
            nb = rx.rx_attn_extend_workspace(max_ctx, max_n, p.hkv, p.d)
            self.ws = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(2)]
        # per-part stores need every new row in exactly one part
        self.split_store = covered == n_new
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.s_comp2 = torch.cuda.Stream()

    def bytes_in(self):
        return sum(h.numel() * h.element_size() for h in self.h_in)

    def bytes_out(self):
        return sum(h.numel() * h.element_size() for h in self.h_out)

    def _copy_rows(self, a, b):
        st = self.st
        st.k_new[a:b].copy_(self.h_k[a:b], non_blocking=True)
        st.v_new[a:b].copy_(self.h_v[a:b], non_blocking=True)
        st.slots[a:b].copy_(self.h_sl[a:b], non_blocking=True)
        if "new" in self.h_pos:
            st.pos_new[a:b].copy_(self.h_pos["new"][a:b], non_blocking=True)

    def _store_rows(self, a, b):
        """Stores new rows a .. b - 1 as the step's store does (bf16 or E4M3
        pools, K rotated on the way in when the step carries RoPE)."""
        st, rx = self.st, self.rx
        if b <= a:
            return
        k, v, sl = st.k_new[a:b], st.v_new[a:b], st.slots[a:b]
        if st.kv_fp8 and st.rope_base:
            rx.rx_kv_store_rope_fp8(st.k8, st.v8, 1.0, 1.0, k, v, sl, st.pos_new[a:b], st.rope_base, st.status)
        elif st.kv_fp8:
            rx.rx_kv_store_fp8(st.k8, st.v8, 1.0, 1.0, k, v, sl, st.status)
        elif st.rope_base:
            rx.rx_kv_store_rope(st.k_pool, st.v_pool, k, v, sl, st.pos_new[a:b], st.rope_base, st.status)
        else:
            rx.rx_kv_store(st.k_pool, st.v_pool, k, v, sl, st.status)

    def load_inputs(self):
        """The step's inputs copied in from the host buffers, in order."""
        st = self.st
        self._copy_rows(0, len(st.prob.new_slots))
        if st.has_dec:
            st.q_dec.copy_(self.h_qd[0])
            st.dec_len.copy_(self.h_qd[1])
        if st.has_ext:
            st.q_ext.copy_(self.h_qe)
        for k, t in (("dec", "pos_dec"), ("ext", "pos_ext")):
            if k in self.h_pos:
                getattr(st, t).copy_(self.h_pos[k])

    def step(self):
        torch, rx, st, p = self.torch, self.rx, self.st, self.st.prob
        E = torch.cuda.Event
        comp = torch.cuda.current_stream()
        split = self.split_store
        ev_dec, ev_dec_rows = E(), E()
        ev_c = [E() for _ in self.chunks]
        ev_c_rows = [E() for _ in self.chunks]   # a part's new rows are in: its store may start
        # the side streams fork from the compute stream (required when captured)
        self.s_in.wait_stream(comp)
        self.s_out.wait_stream(comp)
        self.s_comp2.wait_stream(comp)
        with torch.cuda.stream(self.s_in):
            if split:
                self._copy_rows(*self.dec_rows)
            else:
                self._copy_rows(0, len(p.new_slots))
            ev_dec_rows.record()
            if st.has_dec:
                st.q_dec.copy_(self.h_qd[0], non_blocking=True)
                st.dec_len.copy_(self.h_qd[1], non_blocking=True)
                if "dec" in self.h_pos:
                    st.pos_dec.copy_(self.h_pos["dec"], non_blocking=True)
            ev_dec.record()
            for c, ev, ev_r in zip(self.chunks, ev_c, ev_c_rows):
                if split:
                    self._copy_rows(*c["kv"])
                ev_r.record()
                r0, r1 = c["rows"]
                st.q_ext[r0:r1].copy_(self.h_qe[r0:r1], non_blocking=True)
                if "ext" in self.h_pos:
                    st.pos_ext[r0:r1].copy_(self.h_pos["ext"][r0:r1], non_blocking=True)
                ev.record()
        # each store runs as soon as its rows are in, while its queries arrive
        comp.wait_event(ev_dec_rows)
        if split:
            self._store_rows(*self.dec_rows)
        else:
            st.store_fp8() if st.kv_fp8 else st.kv_store()
        comp.wait_event(ev_dec)
        if st.has_dec:
            if st.rope_base:
                rx.rx_rope(st.q_dec, st.pos_dec, st.rope_base)
            st.decode()
            ev_d = E()
            ev_d.record(comp)
            self.s_out.wait_event(ev_d)
            with torch.cuda.stream(self.s_out):
                self.h_od.copy_(st.o_dec, non_blocking=True)
        # the chunks alternate between two compute streams: the requests of
        # different chunks read and write disjoint rows and slots, so one
        # chunk's staging and last wave overlap the next chunk's attention
        streams = (comp, self.s_comp2)
        for i, (c, ev, ev_r) in enumerate(zip(self.chunks, ev_c, ev_c_rows)):
            r0, r1 = c["rows"]
            cs = streams[i % 2]
            cs.wait_event(ev_r)
            with torch.cuda.stream(cs):
                if split:
                    self._store_rows(*c["kv"])
            cs.wait_event(ev)
            with torch.cuda.stream(cs):
                if st.rope_base:
                    rx.rx_rope(st.q_ext[r0:r1], st.pos_ext[r0:r1], st.rope_base)
                if st.kv_fp8:
                    rx.rx_attn_extend_fp8(st.k8, st.v8, 1.0, 1.0, st.q_ext[r0:r1], st.o_ext[r0:r1], None,
                                          c["qo"], c["req"], c["P"], c["E"], st.rtt, c["max_E"], p.sm_scale,
                                          self.ws[i % 2], st.status, stream=cs)
                else:
                    rx.rx_attn_extend(st.k_pool, st.v_pool, st.q_ext[r0:r1], st.o_ext[r0:r1], None, c["qo"],
                                      c["req"], c["P"], c["E"], st.rtt, c["max_E"], p.sm_scale, st.status,
                                      workspace=self.ws[i % 2], stream=cs)
            ev_o = E()
            ev_o.record(cs)
            self.s_out.wait_event(ev_o)
            with torch.cuda.stream(self.s_out):
                self.h_oe[r0:r1].copy_(st.o_ext[r0:r1], non_blocking=True)
        # the side streams join the compute stream (required when captured)
        comp.wait_stream(self.s_comp2)
        comp.wait_stream(self.s_in)
        comp.wait_stream(self.s_out)

    def capture(self):
        """The step as one CUDA graph (copies, kernels and the events between
        them); replaying it re-issues the same calls without host work."""
        torch = self.torch
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()


def run_e2e(st, torch, rx, steps, flush, dist=None, world=1):
    """The step as a caller runs it through the public API, one step at a
    time: the step's inputs copied in from pinned host memory (new K/V rows
    and their slots, the queries, the decode lengths), the path, its outputs
    copied back, and a synchronize -- a serving loop reads every step's
    output before it can form the next step.  Host wall time per step, L2
    flushed (untimed) before each one.  The copies overlap the kernels
    (E2EPipeline), on bf16 or FP8 pools, with or without RoPE.  The decode
    plan is not rebuilt per step:
    it was built once for the batch (its time is reported beside), and each
    request's last piece follows its length on the device, so the same plan
    serves the batch's later decode steps."""
    p = st.prob
    pipe = E2EPipeline(st, torch, rx)
    h2d, d2h = pipe.bytes_in(), pipe.bytes_out()
    for _ in range(2):   # untimed: first use of the streams and events
        pipe.step()
    torch.cuda.synchronize()

    def timed(run, n):
        secs = []
        for _ in range(n):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run()
            torch.cuda.synchronize()
            secs.append(time.perf_counter() - t0)
        return sum(secs) / n * 1e3

    eager_ms = timed(pipe.step, max(3, min(steps, 50)))
    pipe.capture()
    run = pipe.graph.replay
    n = max(3, min(steps, 200))
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    ms = max_over_ranks(timed(run, n), dist, "cuda")
    # the overlapped schedule must return what the plain step returns on the
    # same inputs (the step rotates q in place when it carries RoPE)
    got = [h.clone() for h in pipe.h_out]
    pipe.load_inputs()
    st.step()
    torch.cuda.synchronize()
    want = ([st.o_dec.cpu()] if st.has_dec else []) + ([st.o_ext.cpu()] if st.has_ext else [])
    if not all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(got, want)):
        raise RuntimeError("the overlapped end-to-end step returned other outputs than the step")
    _, unit, per_step = step_metric(p)
    out = {"value": round(job_throughput(per_step, world, 1, ms), 3), "unit": unit,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 5),
           "steps": n, "timing": "host wall clock per step, synchronized every step",
           "schedule": "; ".join(["copies on their own streams, overlapping the kernels"] +
                                 (["decode's rows and queries first"] if st.has_dec and pipe.chunks else []) +
                                 ([f"extend in {len(pipe.chunks)} request chunks (" +
                                   ", ".join(str(c["n"]) for c in pipe.chunks) +
                                   " requests) alternating over two compute streams"]
                                  if pipe.chunks else []) +
                                 (["each part stores its own new rows"] if pipe.split_store and pipe.chunks else
                                  [] if pipe.split_store else ["every new row stored first"])),
           "launch": "the step's calls captured once in a CUDA graph, replayed per step",
           "eager": {"ms_per_step": round(eager_ms, 5),
                     "value": round(job_throughput(per_step, world, 1, eager_ms), 3),
                     "launch": "the same calls made directly every step"}}
    if st.has_dec:
        out["decode_plan"] = {"built": "once per batch, reused by every later decode step",
                              "build_ms": round(st.plan_build_ms, 3)}
    return out


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# a part's main kernel, from one ncu capture of that kernel alone; each entry
# says which capture.  An entry is removed whenever its kernel changes, so
# that an old count is never reported for new code.
PROFILED_TRAFFIC = {
    ("mixed_chat", "staged"): (
        846_800_000, "ncu --set full -k extend_kernel -c 1 on mixed_chat (600,000-slot pool; the kernel "
                     "reads the same staged rows, Q and O at any pool size): extend_kernel alone"),
    ("mixed_chat", "decode"): (
        1_649_400_000, "ncu --set full -k decode_gqa_kernel -c 1 on mixed_chat (600,000-slot pool; "
                       "same rows; 240 private pieces and 152 group items, longest first; private rows "
                       "evict-first, partials evict-last): decode_gqa_kernel alone, without the merge"),
    ("few_shot_decode", "decode"): (
        290_300_000, "ncu --set full -k decode_kernel -c 1 and -k decode_wide_kernel -c 1 on few_shot_decode "
                     "(262,144-slot pool; same rows; private rows evict-first, partials evict-last): the two "
                     "decode kernels, without the merge"),
    ("tree_of_thought_decode", "decode"): (
        364_000_000, "ncu --set full -k decode_gqa_kernel -c 1 on tree_of_thought_decode (131,072-slot pool; "
                     "same rows; private ranges whole, 4 parts a row, items longest first, private rows "
                     "evict-first, partials evict-last): decode_gqa_kernel alone, without the merge"),
    ("cached_prefix_extend", "staged"): (
        374_900_000, "ncu --set full -k extend_kernel -c 1 on cached_prefix_extend (36,000-slot pool; same "
                     "staged rows, shared prefix tiles staged once): extend_kernel alone, without the "
                     "staging copy"),
    ("constrained_decode", "fsm"): (
        135_200_000, "ncu --set full -k fsm_scan_kernel -c 1 on constrained_decode: the scan (32-bit value keys "
                     "per thread) with the finish in its last CTA (the whole step)"),
    # FP8 (E4M3) pools (--kv-fp8)
    ("few_shot_decode", "decode_fp8"): (
        147_500_000, "ncu --set full -k decode_kernel -c 1 and -k decode_wide_kernel -c 1 on few_shot_decode "
                     "--kv-fp8 (262,144-slot pool; same rows; private rows evict-first, partials evict-last): the "
                     "two FP8 decode kernels, without the merge"),
    ("tree_of_thought_decode", "decode_fp8"): (
        184_700_000, "ncu --set full -k decode_gqa_kernel -c 1 on tree_of_thought_decode --kv-fp8 (131,072-slot "
                     "pool; same rows; private rows evict-first, partials evict-last): decode_gqa_kernel<F8> "
                     "alone, without the merge"),
    ("mixed_chat", "decode_fp8"): (
        827_500_000, "ncu --set full -k decode_gqa_kernel -c 1 on mixed_chat --kv-fp8 (600,000-slot pool; same "
                     "rows; private rows evict-first, partials evict-last): decode_gqa_kernel<F8> alone, without "
                     "the merge"),
    ("cached_prefix_extend", "staged_fp8"): (
        375_100_000, "ncu --set full -k extend_kernel -c 1 on cached_prefix_extend --kv-fp8 (36,000-slot pool; "
                     "same staged rows): extend_kernel alone, without the staging copy"),
    ("mixed_chat", "staged_fp8"): (
        846_800_000, "ncu --set full -k extend_kernel -c 1 on mixed_chat --kv-fp8 (600,000-slot pool; same "
                     "staged rows): extend_kernel alone, without the staging copy"),
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
    """Compact host pools for the oracle: the cached rows in the order they
    were drawn, then the step's new rows placed by the oracle's own
    kv_store, and req_to_token renamed to those rows (pool rows renamed
    consistently give the same attention)."""
    import oracle
    S = prob.num_slots
    row_of = np.full(S, -1, np.int64)
    nc = len(prob.cached_slots)
    row_of[prob.cached_slots] = np.arange(nc)
    fresh = prob.new_slots[row_of[prob.new_slots] < 0]
    row_of[fresh] = nc + np.arange(len(fresh))
    kp = np.zeros((nc + len(fresh), prob.hkv, prob.d), np.uint16)
    vp = np.zeros_like(kp)
    kp[:nc], vp[:nc] = prob.cached_k, prob.cached_v
    oracle.kv_store(kp, vp, prob.new_k, prob.new_v, row_of[prob.new_slots].astype(np.int32))
    rtt = prob.req_to_token
    ok = (rtt >= 0) & (rtt < S)
    rtt_c = np.where(ok, row_of[np.where(ok, rtt, 0)], -1).astype(np.int32)
    return kp, vp, rtt_c


def head_pools(prob, pools):
    """The oracle's pools cut to kv head 0 (each kv head's attention costs
    the same, so the sample runs one and the rate counts the others)."""
    kp, vp, rtt = pools
    return np.ascontiguousarray(kp[:, :1]), np.ascontiguousarray(vp[:, :1]), rtt


def oracle_sample(prob, hp, rows_dec, ext_tokens, threads):
    """One bounded oracle pass on kv head 0 (its G q heads): the first
    rows_dec decode rows, and ext_tokens extend tokens of each extend
    request, evenly spaced over its new tokens (its last token included).
    Returns (decode seconds, rows, extend seconds, tokens, extend flops)."""
    import oracle
    kp, vp, rtt = hp
    G = prob.hq // prob.hkv
    sd = se = 0.0
    nd = ne = flops = 0
    if len(prob.dec_req_idx) and rows_dec:
        nd = min(rows_dec, len(prob.dec_req_idx))
        q = np.ascontiguousarray(prob.q_dec[:nd, :G])
        t0 = time.perf_counter()
        oracle.decode(q, kp, vp, rtt, prob.dec_req_idx[:nd], prob.dec_seq_len[:nd], prob.sm_scale,
                      n_threads=threads)
        sd = time.perf_counter() - t0
    if len(prob.ext_req_idx) and ext_tokens:
        q_rows, kend, qi = [], [], []
        for b in range(len(prob.ext_req_idx)):
            E, P = int(prob.ext_extend_len[b]), int(prob.ext_prefix_len[b])
            k = min(E, ext_tokens)
            for i in sorted({E - 1 - (j * E) // k for j in range(k)}):
                qi.append(int(prob.qo_indptr[b]) + i)
                q_rows.append(int(prob.ext_req_idx[b]))
                kend.append(P + i + 1)
        kend = np.array(kend, np.int32)
        q = np.ascontiguousarray(prob.q_ext[qi][:, :G])
        t0 = time.perf_counter()
        oracle.attention(q, kp, vp, rtt, np.array(q_rows, np.int32), np.zeros_like(kend), kend, prob.sm_scale,
                         n_threads=threads)
        se = time.perf_counter() - t0
        ne = len(kend)
        flops = int(4 * prob.d * G * kend.astype(np.int64).sum())
    return sd, nd, se, ne, flops


def _sample_shape(prob, frac, threads=1):
    """(decode rows, extend tokens per request) for a fraction of the step;
    at least one decode row per thread (the oracle spreads rows, not a
    row's keys, over its threads)."""
    nd = len(prob.dec_req_idx)
    emax = int(prob.ext_extend_len.max()) if len(prob.ext_req_idx) else 0
    rows = min(nd, max(threads, int(np.ceil(nd * frac)))) if nd else 0
    toks = min(emax, max(1, int(np.ceil(emax * frac)))) if emax else 0
    return rows, toks


class OracleRate:
    """Accumulates oracle samples; the rate is the step's own mix of decode
    rows and extend tokens (or its flops), at the measured time per decode
    row and per extend token, over all kv heads."""

    def __init__(self, prob):
        self.prob = prob
        self.sd = self.se = 0.0
        self.nd = self.ne = self.flops = 0

    def add(self, sample):
        sd, nd, se, ne, fl = sample
        self.sd, self.nd, self.se, self.ne, self.flops = (self.sd + sd, self.nd + nd, self.se + se,
                                                          self.ne + ne, self.flops + fl)

    def seconds(self):
        return self.sd + self.se

    def value(self):
        p = self.prob
        _, unit, per_step = step_metric(p)
        if unit == "TFLOP/s":
            return self.flops / self.se / 1e12          # head 0's flops over head 0's time
        t_row = self.sd / self.nd * p.hkv if self.nd else 0.0
        t_tok = self.se / self.ne * p.hkv if self.ne else 0.0
        n_dec, n_ext = len(p.dec_req_idx), int(np.sum(p.ext_extend_len))
        return per_step / (n_dec * t_row + n_ext * t_tok)


def _describe(prob, name, rows, toks):
    parts = []
    if rows:
        parts.append(f"{rows} of {len(prob.dec_req_idx)} decode rows")
    if toks:
        parts.append(f"{toks} of each extend request's {int(prob.ext_extend_len.max())} new tokens "
                     f"(evenly spaced, last included) over {len(prob.ext_req_idx)} requests")
    return (" + ".join(parts) + f" of {name}, on kv head 0 of {prob.hkv} (fp64); the rate weighs "
            "decode rows and extend tokens as the step does and counts every kv head")


def calibrated_sample(prob, hp, threads, seconds):
    """The fraction of a step whose oracle pass takes about `seconds`."""
    frac = 1.0 / 1024
    while True:
        rows, toks = _sample_shape(prob, frac, threads)
        sd, _, se, _, _ = oracle_sample(prob, hp, rows, toks, threads)
        sec = sd + se
        if sec >= seconds / 8 or frac >= 1.0:
            return min(1.0, frac * max(1.0, seconds / max(sec, 1e-4)))
        frac = min(1.0, frac * 4)


def cpu_rate(prob, name, hp, threads, budget_s):
    """The oracle as it stands on `threads` host cores, repeated over a
    bounded sample of the step until about budget_s seconds of CPU work."""
    frac = calibrated_sample(prob, hp, threads, budget_s / 3)
    rows, toks = _sample_shape(prob, frac, threads)
    acc, reps = OracleRate(prob), 0
    while acc.seconds() < budget_s and reps < 10000:
        acc.add(oracle_sample(prob, hp, rows, toks, threads))
        reps += 1
    _, unit, _ = step_metric(prob)
    return {"value": round(acc.value(), 6), "unit": unit, "cores": threads, "kind": "oracle",
            "sample": _describe(prob, name, rows, toks) + f"; repeated {reps} times",
            "seconds": round(acc.seconds(), 3)}


SINGLE_CORE_WORKLOADS = ("tiny_extend", "few_shot_decode", "tree_of_thought_decode")


def cpu_baseline(prob, name, budget_s=15.0):
    """The oracle on all host cores; for the small and decode configurations
    also on one core."""
    hp = head_pools(prob, _oracle_pools(prob))
    out = cpu_rate(prob, name, hp, cores(), budget_s)
    if name in SINGLE_CORE_WORKLOADS:
        out["single_core"] = cpu_rate(prob, name, hp, 1, budget_s / 2)
    return out


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
                     "kernel": ("rx_fsm_step (fsm_scan_kernel; its last CTA finishes every request)" if B <= 512
                                else "rx_fsm_step (fsm_scan_kernel + fsm_finish_kernel)"),
                     "algorithmic_bytes_per_launch": int(algo),
                     "launch_ms": round(k_ms, 5), "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"},
        "e2e": {"value": round(job_throughput(B, world, n, e2e_ms), 3), "unit": "req/s",
                "h2d_bytes_per_step": int(logits.nbytes + state0.nbytes),
                "d2h_bytes_per_step": int(out.numel() * 4 + cnt.numel() * 4), "ms_per_step": round(e2e_ms / n, 5),
                "steps": n},
        "gpu_launches": (1 if B <= 512 else 2) * args.steps, "clocks": clk.summary(),
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
    hp = head_pools(prob, _oracle_pools(prob))
    # a step = a bounded sample of the workload, sized so that the whole run
    # takes about --cpu-seconds
    budget = max(0.05, args.cpu_seconds / max(1, args.steps + args.warmup))
    frac = calibrated_sample(prob, hp, threads, budget)
    rows, toks = _sample_shape(prob, frac, threads)
    acc = OracleRate(prob)
    for i in range(args.warmup + args.steps):
        sample = oracle_sample(prob, hp, rows, toks, threads)
        if i >= args.warmup:
            acc.add(sample)
    metric, unit, _ = step_metric(prob)
    value = acc.value()
    line = {"impl": "reference", "metric": f"prefix-shared attn: {metric}", "value": round(value, 6),
            "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(acc.seconds() / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, random slot permutation)",
            "config": workload_config(prob, args.workload, world, args.extend_path, getattr(args, "graph", False),
                                      getattr(args, "rope", 0.0)),
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": _describe(prob, args.workload, rows, toks) + "; one sample per step"},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="mixed_chat", choices=WORKLOADS + [FSM_WORKLOAD])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool-slots", type=int, default=0,
                    help="override the pool size (profiling runs on a smaller device footprint)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="the step on FP8 (E4M3) pools: K/V rows stored as codes, extend and decode over them")
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
