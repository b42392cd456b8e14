"""Benchmark of the fused FP16 attention hot path on GB300.

One step is one pass of the whole hot path over one batch of synthetic input,
all three variants at full size:
  * dense video attention      B1 H24 S32768 D128                (attn_dense_fwd)
  * VSA                         B1 H24 S32768 D128, 512 cubes, top-64
                                (vsa_select_blocks + vsa_pair_query_cubes + vsa_sparse_fwd)
  * paged E4M3 long prefill     Hq6 Hkv1 D256, Q=8192 after KV=131072
                                (e4m3_paged_to_fp16 + attn_causal_prefill_fwd)
The metric is useful attention TFLOP/s (4 * D * visible (query, key) pairs per
head; VSA counts only the selected cubes) with the bridge's HBM GB/s beside it.
Inputs are seeded synthetic data resident in HBM before the timed region; each
step touches about 1.7 GB, more than the 129 MB L2, so no explicit L2 flush is
done between steps.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
        [--workload all|dense_video|vsa_video|paged_e4m3|dense_small|causal_small]
        [--decode on|off|only] [--masked on|off|only] [--vsa-full on|off|only]
        [--paged-fused on|off|only]
Beside the step, the paged E4M3 decode (4 ragged sequences of 65571..131072
cached tokens, Hq6 Hkv1 D256, one new token each; attn_paged_decode_fwd) is
timed on its own and reported as "decode" with its HBM roofline, and dense attention
with an additive mask (B1 H24 S8192 D128, one FP16 [8192][8192] mask shared by the
heads; attn_dense_mask_fwd) as "masked", and the full VSA layout (1024 prefix
tokens + an 8x62x62 grid with padded boundary cubes; vsa_select_blocks +
vsa_sparse_fwd with prefix and cube counts) as "vsa_full".
For N > 1 (torchrun, one process per GPU) every rank runs the same step on its
own GPU (independent replicas, no data-path communication); the time is the
maximum over ranks and the value counts the work of all ranks.
"""

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_fp16_flashattention_gb300 import inputs  # noqa: E402

PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------ work model
def dense_flops(B, H, Sq, Skv, D):
    return 4.0 * B * H * Sq * Skv * D


def causal_pairs(Q, KV):
    prefix = KV - Q
    return Q * prefix + Q * (Q + 1) // 2


def causal_flops(B, Hq, Q, KV, D):
    return 4.0 * D * B * Hq * causal_pairs(Q, KV)


def vsa_flops(B, H, S, D, topk, block=64):
    return 4.0 * B * H * S * topk * block * D


def bridge_bytes(KV, Hkv, D, page_size):
    n_pages = -(-KV // page_size)
    return 2 * KV * Hkv * D + 4 * n_pages + 2 * 2 * KV * Hkv * D


def decode_bytes(kv_lens, B, Hq, Hkv, nq, D, page_size):
    """Bytes a paged decode must move: every live K and V byte, the page-table
    entries it reads, Q and the FP16 output (lengths and lse are negligible)."""
    tokens = int(sum(kv_lens))
    pages = int(sum(-(-n // page_size) for n in kv_lens))
    return 2 * tokens * Hkv * D + 4 * pages + 2 * (2 * B * Hq * nq * D)


# ------------------------------------------------------------------ workloads on the GPU
class Workload:
    """Device-resident inputs and outputs of one sub-workload plus its calls."""

    def __init__(self, name, gb, torch, dev, host_inputs):
        self.name, self.gb, self.torch, self.dev = name, gb, torch, dev
        w = inputs.WORKLOADS[name]
        self.w = w
        self.host = host_inputs
        T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        if w["kind"] == "dense":
            self.q, self.k, self.v = (T(x) for x in host_inputs)
            self.o = torch.empty_like(self.q)
            self.flops = dense_flops(w["B"], w["H"], w["S"], w["S"], w["D"])
        elif w["kind"] == "causal":
            self.q, self.k, self.v = (T(x) for x in host_inputs)
            self.o = torch.empty_like(self.q)
            ws = gb.attn_causal_prefill_workspace_size(w["B"], w["Hq"], w["Q"], w["KV"], w["D"])
            self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
            self.flops = causal_flops(w["B"], w["Hq"], w["Q"], w["KV"], w["D"])
        elif w["kind"] == "vsa":
            self.q, self.k, self.v = (T(x) for x in host_inputs)
            S = self.q.shape[2]
            nc = S // 64
            self.idx = torch.empty((w["B"], w["H"], nc, w["topk"]), dtype=torch.int32, device=dev)
            self.pairs = torch.empty((w["B"], w["H"], (nc + 1) // 2, 2), dtype=torch.int32,
                                     device=dev)
            ws = gb.vsa_select_workspace_size(w["B"], w["H"], S, w["D"], 64)
            self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
            self.pair_ws = torch.empty(gb.load().vsa_pair_workspace_size(w["B"], w["H"], nc),
                                       dtype=torch.uint8, device=dev)
            self.counter = torch.zeros(gb.load().vsa_sparse_workspace_size(), dtype=torch.uint8,
                                       device=dev)
            self.o = torch.empty_like(self.q)
            self.flops = vsa_flops(w["B"], w["H"], S, w["D"], w["topk"])
        elif w["kind"] == "paged":
            qh, kp, vp, table = host_inputs
            self.q, self.kp, self.vp, self.table = T(qh), T(kp), T(vp), T(table)
            self.kf = torch.empty((w["Hkv"], w["KV"], w["D"]), dtype=torch.float16, device=dev)
            self.vf = torch.empty_like(self.kf)
            self.o = torch.empty_like(self.q)
            ws = gb.attn_causal_prefill_workspace_size(w["B"], w["Hq"], w["Q"], w["KV"], w["D"])
            self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
            self.flops = causal_flops(w["B"], w["Hq"], w["Q"], w["KV"], w["D"])
            self.bridge_bytes = bridge_bytes(w["KV"], w["Hkv"], w["D"], w["page_size"])

    def calls(self):
        """(label, fn) pairs in launch order; each fn queues GPU work on the current stream."""
        gb, w = self.gb, self.w
        if w["kind"] == "dense":
            return [("attn_dense_fwd", lambda: gb.attn_dense_fwd(self.q, self.k, self.v, o=self.o))]
        if w["kind"] == "causal":
            return [("attn_causal_prefill_fwd",
                     lambda: gb.attn_causal_prefill_fwd(self.q, self.k, self.v, o=self.o,
                                                        workspace=self.ws))]
        if w["kind"] == "vsa":
            return [("vsa_select_blocks",
                     lambda: gb.vsa_select_blocks(self.q, self.k, w["topk"], idx=self.idx,
                                                  workspace=self.ws)),
                    ("vsa_pair_query_cubes",
                     lambda: gb.vsa_pair_query_cubes(self.idx, pairs=self.pairs,
                                                     workspace=self.pair_ws)),
                    ("vsa_sparse_fwd",
                     lambda: gb.vsa_sparse_fwd(self.q, self.k, self.v, self.idx, pairs=self.pairs,
                                               o=self.o, workspace=self.counter))]
        return [("e4m3_paged_to_fp16",
                 lambda: gb.e4m3_paged_to_fp16(self.kp, self.vp, self.table, w["KV"], w["k_scale"],
                                               w["v_scale"], k_out=self.kf, v_out=self.vf)),
                ("attn_causal_prefill_fwd(paged)",
                 lambda: gb.attn_causal_prefill_fwd(self.q, self.kf[None], self.vf[None], o=self.o,
                                                    workspace=self.ws, prob_split=True))]

    # host <-> device traffic of the end-to-end variant
    def h2d_pairs(self):
        if self.w["kind"] == "paged":
            return [(self.q, 0), (self.kp, 1), (self.vp, 2), (self.table, 3)]
        return [(self.q, 0), (self.k, 1), (self.v, 2)]

    def d2h(self):
        out = [self.o]
        if self.w["kind"] == "vsa":
            out.append(self.idx)
        return out


def host_inputs(name):
    w = inputs.WORKLOADS[name]
    if w["kind"] == "dense":
        return inputs.dense_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"], video=w.get("video", False))
    if w["kind"] == "causal":
        return inputs.causal_inputs(w["B"], w["Hq"], w["Hkv"], w["Q"], w["KV"], w["D"], w["seed"])
    if w["kind"] == "vsa":
        return inputs.vsa_inputs(w["B"], w["H"], w["D"], w["seed"], w["grid"], w["cube"])
    q = inputs.causal_inputs(w["B"], w["Hq"], w["Hkv"], w["Q"], 32, w["D"], w["seed"])[0]
    kp, vp, table = inputs.paged_e4m3_inputs(w["Hkv"], w["KV"], w["D"], w["seed"], w["page_size"])
    return q, kp, vp, table


# ------------------------------------------------------------------ clocks
CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi samples every 50 ms, started before the warm-up so that it is
    running when the timed region begins; only samples stamped inside the
    window given to stop() are summarised."""

    def __init__(self, gpu_index, path=None):
        self.proc = None
        self.gpu = gpu_index
        self.path = path or os.path.join(tempfile.gettempdir(),
                                         f"gbattn_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            return summarize_clocks(fh.read().splitlines(), window)


def summarize_clocks(lines, window=None):
    """Median SM clock, maximum clock and active throttle reasons of nvidia-smi CSV
    lines (CLOCK_QUERY order), over the samples stamped inside `window` (all if
    none is) and drawing more than 200 W (all if none does)."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
        except ValueError:
            when = None   # unknown stamp format: the sample is kept
        try:
            rows.append(dict(t=when, sm=float(parts[2]), max=float(parts[3]),
                             power=float(parts[4]), hw=parts[6], hwt=parts[7], swt=parts[8],
                             swp=parts[9]))
        except ValueError:
            continue
    if window is not None:
        inside = [r for r in rows if r["t"] is None or window[0] <= r["t"] <= window[1]]
        rows = inside or rows
    if not rows:
        return None
    loaded = [r for r in rows if r["power"] > 200.0] or rows
    reasons = set()
    for r in loaded:
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
            "sm_max_mhz": max(r["max"] for r in loaded),
            "samples": len(loaded), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], tc=p.get("bf16_tflops"), tc_sust=p.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sust=1700.0, src="fallback")


KERNEL_SOURCES = {
    "attn_dense_kernel": ("attn_dense.cu", "ptx.cuh", "host.h"),
    "attn_fwd_kernel<128,sparse>": ("attn.cu", "ptx.cuh", "host.h"),
    "attn_fwd_kernel<256,causal>+merge": ("attn.cu", "ptx.cuh", "host.h"),
    "e4m3_bridge_kernel": ("bridge.cu", "e4m3.cuh", "ptx.cuh", "host.h"),
    "paged_decode_kernel+merge": ("decode.cu", "e4m3.cuh", "ptx.cuh", "host.h"),
    "attn_fwd_kernel<128,masked>": ("attn.cu", "ptx.cuh", "host.h"),
}


def source_sha(kernel):
    """Hash of the source files a kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_fp16_flashattention_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel):
    """DRAM bytes per launch from the committed ncu capture, if the kernel's sources are unchanged."""
    if not os.path.exists(PROFILE_TRAFFIC) or kernel not in KERNEL_SOURCES:
        return None
    t = json.load(open(PROFILE_TRAFFIC))
    e = t.get(kernel)
    if not e or e.get("source_sha") != source_sha(kernel):
        return None
    return e.get("bytes_per_launch")


def physical_gpu_index(local):
    """nvidia-smi index of this process's GPU (CUDA_VISIBLE_DEVICES maps local ordinals)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        import torch
        if not torch.cuda.is_available():
            backend = "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(value, world, device=None):
    """Maximum of a float over all ranks (host-side bookkeeping only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ oracle timing (CPU)
def oracle_sample(names, budget_s=20.0):
    """Time the CPU oracle on a bounded sample of every sub-workload (rows of the
    attention outputs; the selection and bridge are not part of the TFLOP/s figure).
    Returns (useful_flops_done, seconds, description)."""
    from oracle import attention as OA
    from oracle import e4m3 as OE
    from oracle import vsa as OV
    done = 0.0
    secs = 0.0
    desc = []
    share = budget_s / max(1, len(names))
    for name in names:
        w = inputs.WORKLOADS[name]
        data = host_inputs(name)
        rows_done = 0
        t_used = 0.0
        n = 16
        while t_used < share:
            if w["kind"] == "dense":
                q, k, v = data
                rows = inputs.sample_rows(w["B"] * w["H"], w["S"], n, seed=9000 + rows_done)
                t0 = time.perf_counter()
                OA.dense_attention(q, k, v, inputs.softmax_scale(w["D"]), rows=rows)
                t_used += time.perf_counter() - t0
                done += n * 4.0 * w["S"] * w["D"]
            elif w["kind"] == "vsa":
                q, k, v = data
                if rows_done == 0:
                    t0 = time.perf_counter()
                    idx = OV.vsa_select(q, k, 64, w["topk"])
                    t_used += time.perf_counter() - t0
                rows = inputs.sample_rows(w["B"] * w["H"], q.shape[2], n, seed=9000 + rows_done)
                t0 = time.perf_counter()
                OA.vsa_sparse_attention(q, k, v, idx, 64, inputs.softmax_scale(w["D"]), rows=rows)
                t_used += time.perf_counter() - t0
                done += n * 4.0 * w["topk"] * 64 * w["D"]
            elif w["kind"] in ("paged", "causal"):
                if w["kind"] == "paged":
                    q, kp, vp, table = data
                    if rows_done == 0:
                        t0 = time.perf_counter()
                        kb, vb = OE.paged_e4m3_to_fp16(kp, vp, table, w["KV"], w["k_scale"],
                                                       w["v_scale"])
                        k, v = kb.view(np.float16)[None], vb.view(np.float16)[None]
                        t_used += time.perf_counter() - t0
                else:
                    q, k, v = data
                rows = inputs.sample_rows(w["B"] * w["Hq"], w["Q"], n, seed=9000 + rows_done)
                t0 = time.perf_counter()
                OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(w["D"]), w["Q"], rows=rows)
                t_used += time.perf_counter() - t0
                prefix = w["KV"] - w["Q"]
                done += 4.0 * w["D"] * float(np.sum(prefix + rows[:, 1] + 1))
            rows_done += n
            n = min(n * 2, 256)
        secs += t_used
        desc.append(f"{name}: {rows_done} sampled rows")
    return done, secs, "; ".join(desc)


# ------------------------------------------------------------------ main
def run_reference(args, names, world, rank):
    """The oracle as it stands, on the host cores, same metric and config."""
    if rank != 0:
        return 0
    per_step = []
    done_total = 0.0
    for _ in range(args.warmup):
        oracle_sample(names, budget_s=2.0)
    desc = ""
    for _ in range(args.steps):
        done, secs, desc = oracle_sample(names, budget_s=args.ref_budget)
        per_step.append((done, secs))
        done_total += done
    tflops = sum(d for d, _ in per_step) / sum(s for _, s in per_step) / 1e12
    ms = 1e3 * sum(s for _, s in per_step) / len(per_step)
    line = {"metric": "attention useful TFLOP/s", "value": tflops, "unit": "TFLOP/s",
            "impl": "reference", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": "+".join(names), "timing": "host wall clock, oracle on CPU"},
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def measure_decode(gb, torch, dev, steps, warmup, pk):
    """Paged E4M3 decode (4 ragged sequences, one new token each), timed on its own.

    Each launch is bracketed by CUDA events on the launching stream.  The 214 MB
    page pool is larger than L2, so launches run back to back; the same launch
    with a 256 MB buffer rewritten before it is reported as well."""
    w = inputs.WORKLOADS["paged_decode"]
    q, kp, vp, table, lens = inputs.paged_decode_inputs(w["B"], w["Hq"], w["Hkv"], w["nq"],
                                                        w["kv_lens"], w["D"], w["seed"],
                                                        w["page_size"])
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    dq, dk, dv, dt, dl = T(q), T(kp), T(vp), T(table), T(lens)
    o = torch.empty_like(dq)
    max_kv = int(max(w["kv_lens"]))
    ws = torch.empty(max(16, gb.attn_paged_decode_workspace_size(w["B"], w["Hq"], w["Hkv"],
                                                                 w["nq"], max_kv, w["D"])),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        gb.attn_paged_decode_fwd(dq, dk, dv, dt, dl, w["k_scale"], w["v_scale"],
                                 max_kv_len=max_kv, o=o, workspace=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    # A serving loop replays its decode step as a CUDA graph; time the call that way
    # (both launches, with the merge's programmatic dependency, in one graph).
    graph = torch.cuda.CUDAGraph()
    n0 = gb.launch_count()
    with torch.cuda.graph(graph):
        call()
    launches = gb.launch_count() - n0
    graph.replay()
    torch.cuda.synchronize()
    def replays(flush_between):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            if flush_between:
                flush.fill_(1)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    # The page pool (214 MB) is larger than L2 and each call reads it once in a fixed
    # order, so back-to-back calls find almost none of it in L2 (ncu: 205 MB of DRAM
    # reads per call); that is the number reported.  Rewriting a 256 MB buffer between
    # calls instead leaves L2 full of dirty lines whose write-back then falls inside
    # the timed call; that figure is reported beside it.
    ms = replays(False)
    ms_flushed = replays(True)
    # Calls back to back in one graph (as consecutive decode steps of a serving loop
    # run): the per-replay graph launch is paid once for 20 calls.
    n_b2b = 20
    graph20 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph20):
        for _ in range(n_b2b):
            call()
    graph20.replay()
    torch.cuda.synchronize()
    evs20 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(max(3, steps // 4))]
    for e0, e1 in evs20:
        e0.record(stream)
        graph20.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_b2b = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs20) / n_b2b
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the decode measurement")
    nbytes = decode_bytes(w["kv_lens"], w["B"], w["Hq"], w["Hkv"], w["nq"], w["D"],
                          w["page_size"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "paged_decode_kernel+merge", "bound": "hbm", "achieved": gbs,
            "unit": "GB/s", "peak": pk["hbm"], "frac": gbs / pk["hbm"],
            "peak_source": f"{pk['src']} HBM copy bandwidth", "ms_per_launch": ms,
            "new_tokens_per_s": w["B"] * w["nq"] / (ms * 1e-3), "bytes_per_launch": nbytes,
            "launches_per_call": launches, "traffic": traffic_for("paged_decode_kernel+merge"),
            "config": {k: v for k, v in w.items() if k != "seed"},
            "timing": "CUDA-graph replay of one attn_paged_decode_fwd call, events around each replay",
            "l2": "page pool larger than L2, calls back to back (no flush)",
            "ms_per_launch_l2_flushed": ms_flushed,
            "frac_l2_flushed": nbytes / (ms_flushed * 1e-3) / 1e9 / pk["hbm"],
            "back_to_back": {"ms_per_launch": ms_b2b,
                             "achieved": nbytes / (ms_b2b * 1e-3) / 1e9,
                             "frac": nbytes / (ms_b2b * 1e-3) / 1e9 / pk["hbm"],
                             "timing": f"CUDA-graph replay of {n_b2b} calls in a row"}}


def bridge_back_to_back(torch, w, n=20, reps=5):
    """Per-call ms of the E4M3 bridge alone, n calls in a row replayed as one CUDA
    graph (median of reps).  Each call's 134 MB of FP16 output is still being
    written back from L2 while the next call runs, as in a steady stream of them;
    inside the step the call instead follows another workload's kernels."""
    fn = dict(w.calls())["e4m3_paged_to_fp16"]
    fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(n):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for e0, e1 in evs:
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if w.gb.device_status() != 0:
        raise RuntimeError("device status flags set during the bridge measurement")
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / n


def measure_small(gb, torch, dev, name, steps, warmup, pk, n=20):
    """One of the two small configurations (dense_small, causal_small), timed on its own.

    A call at these sizes takes tens of microseconds, about as long as the host
    takes to issue it, so it is timed the way a serving loop runs it: n calls in a
    row captured once as a CUDA graph, replayed `steps` times with CUDA events on
    the launching stream; the per-call time is the replay time / n.  The calls
    bracketed one by one with events (host launch gaps included) are reported
    beside it."""
    w = Workload(name, gb, torch, dev, host_inputs(name))
    (_, fn), = w.calls()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    graph = torch.cuda.CUDAGraph()
    n0 = gb.launch_count()
    with torch.cuda.graph(graph):
        for _ in range(n):
            fn()
    launches = (gb.launch_count() - n0) // n
    graph.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t = [e0.elapsed_time(e1) / n for e0, e1 in evs]
    single = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
    for e0, e1 in single:
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    if gb.device_status() != 0:
        raise RuntimeError(f"device status flags set during the {name} measurement")
    ms = statistics.median(t)
    ms_single = statistics.median(e0.elapsed_time(e1) for e0, e1 in single)
    tflops = w.flops / (ms * 1e-3) / 1e12
    return {"ms": ms, "cv": statistics.pstdev(t) / statistics.mean(t) if len(t) > 1 else 0.0,
            "useful_flop": w.flops, "achieved": tflops, "unit": "TFLOP/s", "peak": pk["tc"],
            "frac": tflops / pk["tc"], "peak_source": f"{pk['src']} bf16 burst (kernel timed alone)",
            "launches_per_call": launches,
            "timing": f"CUDA-graph replay of {n} calls in a row, {steps} replays, median",
            "ms_one_call_with_host_launch": ms_single}


def measure_masked(gb, torch, dev, steps, warmup, pk):
    """Dense attention with an additive mask (B1 H24 S8192 D128, one FP16 mask
    [8192][8192] shared by the heads), timed on its own; useful FLOP count only
    the visible (query, key) pairs.  A 256 MB buffer is rewritten between launches."""
    w = inputs.WORKLOADS["dense_masked"]
    q, k, v = inputs.dense_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"])
    mask = inputs.additive_mask(w["S"], w["S"], w["seed"])
    visible = int(np.isfinite(mask).sum())
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    dq, dk, dv, dm = T(q), T(k), T(v), T(mask)
    o = torch.empty_like(dq)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        gb.attn_dense_mask_fwd(dq, dk, dv, dm, o=o)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    n0 = gb.launch_count()
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    launches = (gb.launch_count() - n0) // steps
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the masked measurement")
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    flops = 4.0 * w["D"] * w["B"] * w["H"] * visible
    tf = flops / (ms * 1e-3) / 1e12
    peak = pk["tc"] or pk["tc_sust"]
    mask_bytes = 2 * w["S"] * w["S"]
    return {"kernel": "attn_fwd_kernel<128,masked>", "bound": "tensor", "achieved": tf,
            "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "peak_source": f"{pk['src']} bf16 burst (kernel timed alone; fp16 dense rate = bf16 rate)",
            "ms_per_launch": ms, "useful_flop": flops, "visible_pairs_per_head": visible,
            "mask_bytes": mask_bytes,
            "mask_read_gbs_if_once_per_head": w["H"] * mask_bytes / (ms * 1e-3) / 1e9,
            "launches_per_call": launches, "traffic": traffic_for("attn_fwd_kernel<128,masked>"),
            "config": {k2: v2 for k2, v2 in w.items() if k2 != "seed"},
            "l2": "256 MB buffer rewritten between launches, outside the timed events"}


def measure_vsa_full(gb, torch, dev, steps, warmup, pk):
    """The full VSA layout (1024 prefix tokens + an 8x62x62 grid in 512 cubes with
    padded boundary cubes, B1 H24 D128, top-64), selection + sparse attention,
    timed on its own.  Useful FLOP count the (query, key) pairs the definition
    visits: prefix rows x every real token, real video rows x the real tokens of
    their selected cubes.  A 256 MB buffer is rewritten between calls."""
    w = inputs.WORKLOADS["vsa_full"]
    q, k, v, valid = inputs.vsa_full_inputs(w["B"], w["H"], w["D"], w["seed"], w["grid"],
                                            w["cube"], w["prefix"])
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    dq, dk, dv, dval = T(q), T(k), T(v), T(valid)
    S = q.shape[2]
    nc = valid.size
    idx = torch.empty((w["B"], w["H"], nc, w["topk"]), dtype=torch.int32, device=dev)
    ws = torch.empty(gb.vsa_select_workspace_size(w["B"], w["H"], S, w["D"], 64), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(dq)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def select():
        gb.vsa_select_blocks(dq, dk, w["topk"], prefix=w["prefix"], cube_valid=dval, idx=idx,
                             workspace=ws)

    pairs = torch.empty((w["B"], w["H"], (nc + 1) // 2, 2), dtype=torch.int32, device=dev)

    def sparse():
        gb.vsa_pair_query_cubes(idx, pairs=pairs)
        gb.vsa_sparse_fwd(dq, dk, dv, idx, prefix=w["prefix"], cube_valid=dval, pairs=pairs, o=o)

    for _ in range(warmup):
        select()
        sparse()
    torch.cuda.synchronize()
    real = int(valid.sum())
    sel = idx.cpu().numpy()                                 # work count only
    visited = w["prefix"] * (w["prefix"] + real) * w["B"] * w["H"]
    visited += int((valid[sel].sum(axis=-1) * valid[None, None, :]).sum())
    flops = 4.0 * w["D"] * visited
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        flush.fill_(1)
        e[0].record(stream)
        select()
        e[1].record(stream)
        sparse()
        e[2].record(stream)
    torch.cuda.synchronize()
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the full-VSA measurement")
    t_sel = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    t_sp = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    tf = flops / ((t_sel + t_sp) * 1e-3) / 1e12
    peak = pk["tc"] or pk["tc_sust"]
    return {"kernel": "vsa_pool+vsa_score+vsa_topk+attn_fwd_kernel<128,sparse_full>", "bound": "tensor",
            "achieved": tf, "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "peak_source": f"{pk['src']} bf16 burst (timed alone; fp16 dense rate = bf16 rate)",
            "ms_select": t_sel, "ms_sparse": t_sp, "sparse_tflops": flops / (t_sp * 1e-3) / 1e12,
            "useful_flop": flops, "real_tokens": real, "slots": S,
            "config": {k2: v2 for k2, v2 in w.items() if k2 != "seed"},
            "l2": "256 MB buffer rewritten between calls, outside the timed events"}


def measure_vsa_coarse(gb, torch, dev, steps, warmup, pk):
    """The VSA workload with the coarse branch: vsa_select_blocks_coarse (selection,
    pooled V, cube-level attention over all key cubes) and the sparse attention
    adding gate * coarse output, beside the selection and sparse attention alone.
    Useful FLOP: the fine branch's selected pairs plus the coarse attention's
    4 * D * cubes^2 per head.  A 256 MB buffer is rewritten between calls."""
    w = inputs.WORKLOADS["vsa_video"]
    q, k, v = host_inputs("vsa_video")
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    dq, dk, dv = T(q), T(k), T(v)
    gate = torch.empty_like(dq).uniform_(-1.0, 1.0)
    B, H, S, D = dq.shape
    nc = S // 64
    idx = torch.empty((B, H, nc, w["topk"]), dtype=torch.int32, device=dev)
    oc = torch.empty((B, H, nc, D), dtype=torch.float32, device=dev)
    pairs = torch.empty((B, H, (nc + 1) // 2, 2), dtype=torch.int32, device=dev)
    ws = torch.empty(gb.vsa_select_coarse_workspace_size(B, H, S, D, 64), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(dq)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    calls = {
        "select_coarse": lambda: gb.vsa_select_blocks_coarse(dq, dk, dv, w["topk"], idx=idx,
                                                             coarse=oc, workspace=ws),
        "select": lambda: gb.vsa_select_blocks(dq, dk, w["topk"], idx=idx, workspace=ws),
        "sparse_gated": lambda: (gb.vsa_pair_query_cubes(idx, pairs=pairs),
                                 gb.vsa_sparse_fwd(dq, dk, dv, idx, pairs=pairs, o=o, coarse=oc,
                                                   gate=gate)),
        "sparse": lambda: (gb.vsa_pair_query_cubes(idx, pairs=pairs),
                           gb.vsa_sparse_fwd(dq, dk, dv, idx, pairs=pairs, o=o)),
    }
    res = {}
    for name, fn in calls.items():
        for _ in range(warmup):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the coarse-branch measurement")
    flops = vsa_flops(B, H, S, D, w["topk"]) + 4.0 * D * nc * nc * B * H
    t = res["select_coarse"] + res["sparse_gated"]
    tf = flops / (t * 1e-3) / 1e12
    peak = pk["tc"] or pk["tc_sust"]
    return {"kernel": "vsa_pool+vsa_score+vsa_topk+vsa_coarse_pv+attn_fwd_kernel<128,sparse>",
            "bound": "tensor", "achieved": tf, "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "peak_source": f"{pk['src']} bf16 burst (timed alone; fp16 dense rate = bf16 rate)",
            "ms_select_coarse": res["select_coarse"], "ms_select": res["select"],
            "ms_sparse_gated": res["sparse_gated"], "ms_sparse": res["sparse"],
            "useful_flop": flops,
            "l2": "256 MB buffer rewritten between calls, outside the timed events"}


def measure_paged_fused(gb, torch, dev, steps, warmup, pk):
    """The paged-E4M3 prefill with the bridge fused into the attention
    (attn_causal_prefill_paged_fwd) beside the two-pass bridge + FP16 prefill,
    on the paged_e4m3 workload; both timed on their own with CUDA events."""
    w = inputs.WORKLOADS["paged_e4m3"]
    q = inputs.causal_inputs(w["B"], w["Hq"], w["Hkv"], w["Q"], 32, w["D"], w["seed"])[0]
    kp, vp, table = inputs.paged_e4m3_inputs(w["Hkv"], w["KV"], w["D"], w["seed"], w["page_size"])
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    dq, dk, dv, dt = T(q), T(kp), T(vp), T(table)
    o = torch.empty_like(dq)
    kf = torch.empty((w["Hkv"], w["KV"], w["D"]), dtype=torch.float16, device=dev)
    vf = torch.empty_like(kf)
    ws = torch.empty(max(16, gb.attn_causal_prefill_workspace_size(w["B"], w["Hq"], w["Q"], w["KV"],
                                                                   w["D"])),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fused(split):
        gb.attn_causal_prefill_paged_fwd(dq, dk, dv, dt, w["KV"], w["k_scale"], w["v_scale"], o=o,
                                         workspace=ws, prob_split=split)

    def two_pass(split):
        gb.e4m3_paged_to_fp16(dk, dv, dt, w["KV"], w["k_scale"], w["v_scale"], k_out=kf, v_out=vf)
        gb.attn_causal_prefill_fwd(dq, kf[None], vf[None], o=o, workspace=ws, prob_split=split)

    def prefill_only(split):
        gb.attn_causal_prefill_fwd(dq, kf[None], vf[None], o=o, workspace=ws, prob_split=split)

    res = {}
    for name, fn, split in (("fused", fused, True), ("bridge_then_prefill", two_pass, True),
                            ("fused_fp16_p", fused, False),
                            ("bridge_then_prefill_fp16_p", two_pass, False),
                            ("prefill", prefill_only, True), ("prefill_fp16_p", prefill_only, False)):
        for _ in range(warmup):
            fn(split)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            e0.record(stream)
            fn(split)
            e1.record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the paged measurement")
    flops = causal_flops(w["B"], w["Hq"], w["Q"], w["KV"], w["D"])
    tf = flops / (res["fused"] * 1e-3) / 1e12
    peak = pk["tc_sust"] or pk["tc"]
    tf_p = lambda key: flops / (res[key] * 1e-3) / 1e12
    return {"kernel": "attn_fwd_kernel<256,causal_paged>+merge", "bound": "tensor", "achieved": tf,
            "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "peak_source": f"{pk['src']} bf16 sustained (fp16 dense rate = bf16 rate)",
            "probabilities": "FP16 hi + lo (the path that meets the stated tolerance); *_fp16_p: "
                             "the pages' single FP16 P",
            "ms_fused": res["fused"], "ms_bridge_then_prefill": res["bridge_then_prefill"],
            "ms_fused_fp16_p": res["fused_fp16_p"],
            "ms_bridge_then_prefill_fp16_p": res["bridge_then_prefill_fp16_p"],
            "prefill_alone": {"ms": res["prefill"], "tflops": tf_p("prefill"),
                              "ms_fp16_p": res["prefill_fp16_p"],
                              "tflops_fp16_p": tf_p("prefill_fp16_p")},
            "config": {k2: v2 for k2, v2 in w.items() if k2 != "seed"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--clock-log", default=None,
                    help="file for the raw nvidia-smi samples of the timed region (default: a temp file)")
    ap.add_argument("--decode", default="on", choices=["on", "off", "only"],
                    help="paged E4M3 decode measured beside the step (only: print just that)")
    ap.add_argument("--masked", default="on", choices=["on", "off", "only"],
                    help="dense attention with an additive mask measured beside the step")
    ap.add_argument("--vsa-full", default="on", choices=["on", "off", "only"],
                    help="the full VSA layout (prefix + boundary cubes) measured beside the step")
    ap.add_argument("--vsa-coarse", default="on", choices=["on", "off", "only"],
                    help="the VSA workload with the coarse (compression) branch")
    ap.add_argument("--paged-fused", default="on", choices=["on", "off", "only"],
                    help="the paged prefill with the bridge fused in, beside bridge + prefill")
    ap.add_argument("--small", default="on", choices=["on", "off"],
                    help="the two small configurations (dense B1 H2 S256, causal Q1024/KV4096)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the head count of the dense/VSA workloads (profiling runs)")
    args = ap.parse_args()
    if args.heads > 0:
        for n in ("dense_video", "vsa_video"):
            inputs.WORKLOADS[n] = dict(inputs.WORKLOADS[n], H=args.heads)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    names = ["dense_video", "vsa_video", "paged_e4m3"] if args.workload == "all" else \
        args.workload.split(",")

    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        r = run_reference(args, names, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return r

    import torch
    import attention_fp16_flashattention_gb300 as gb
    from attention_fp16_flashattention_gb300 import build as gbuild
    if not gbuild.up_to_date() and rank == 0:
        gbuild.build()
    barrier(world)
    gb.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    if args.paged_fused == "only":
        if rank == 0:
            print(json.dumps(dict(metric="fused paged prefill useful TFLOP/s", impl="ours",
                                  n_gpus=world, steps=args.steps, warmup=args.warmup,
                                  **measure_paged_fused(gb, torch, dev, args.steps, args.warmup,
                                                        peaks()))))
        return 0
    if args.vsa_coarse == "only":
        if rank == 0:
            print(json.dumps(dict(metric="VSA with the coarse branch useful TFLOP/s", impl="ours",
                                  n_gpus=world, steps=args.steps, warmup=args.warmup,
                                  **measure_vsa_coarse(gb, torch, dev, args.steps, args.warmup,
                                                       peaks()))))
        return 0
    if args.vsa_full == "only":
        if rank == 0:
            print(json.dumps(dict(metric="full VSA useful TFLOP/s", impl="ours", n_gpus=world,
                                  steps=args.steps, warmup=args.warmup,
                                  **measure_vsa_full(gb, torch, dev, args.steps, args.warmup,
                                                     peaks()))))
        return 0
    if args.masked == "only":
        if rank == 0:
            print(json.dumps(dict(metric="masked dense attention useful TFLOP/s", impl="ours",
                                  n_gpus=world, steps=args.steps, warmup=args.warmup,
                                  **measure_masked(gb, torch, dev, args.steps, args.warmup,
                                                   peaks()))))
        return 0
    if args.decode == "only":
        if rank == 0:
            print(json.dumps(dict(metric="paged decode HBM GB/s", impl="ours", n_gpus=world,
                                  steps=args.steps, warmup=args.warmup,
                                  **measure_decode(gb, torch, dev, args.steps, args.warmup,
                                                   peaks()))))
        return 0

    hosts = {n: host_inputs(n) for n in names}
    wls = [Workload(n, gb, torch, dev, hosts[n]) for n in names]
    calls = [(w, lbl, fn) for w in wls for lbl, fn in w.calls()]

    def step():
        for _, _, fn in calls:
            fn()

    clocks = ClockSampler(physical_gpu_index(local), args.clock_log)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during warm-up")

    # ---- timed region: device time with per-call events on the launching stream
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    launches0 = gb.launch_count()
    t_begin = datetime.datetime.now()
    start.record(stream)
    for s in range(args.steps):
        for c, (_, _, fn) in enumerate(calls):
            ev[s][c][0].record(stream)
            fn()
            ev[s][c][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_end = datetime.datetime.now()
    launches = (gb.launch_count() - launches0) // args.steps
    clock_info = clocks.stop((t_begin, t_end))
    barrier(world, dev)
    local_ms = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(local_ms, world, dev)
    if gb.device_status() != 0:
        raise RuntimeError("device status flags set during the timed region")

    per_call, per_call_cv = {}, {}
    for c, (w, lbl, _) in enumerate(calls):
        t = [ev[s][c][0].elapsed_time(ev[s][c][1]) for s in range(args.steps)]
        per_call[f"{w.name}:{lbl}"] = statistics.median(t)
        per_call_cv[f"{w.name}:{lbl}"] = (statistics.pstdev(t) / statistics.mean(t)
                                          if len(t) > 1 else 0.0)

    flops_step = sum(w.flops for w in wls)
    value = world * flops_step / (ms * 1e-3) / 1e12
    pk = peaks()

    # ---- dominant kernel roofline
    attn_calls = {k: v for k, v in per_call.items()
                  if "select" not in k and "e4m3_paged" not in k and "pair" not in k}
    dom = max(attn_calls, key=attn_calls.get)
    dom_w = next(w for w in wls if dom.startswith(w.name + ":"))
    achieved = dom_w.flops / (attn_calls[dom] * 1e-3) / 1e12
    kernel_name = {"dense": "attn_dense_kernel", "vsa": "attn_fwd_kernel<128,sparse>",
                   "paged": "attn_fwd_kernel<256,causal>+merge",
                   "causal": "attn_fwd_kernel<256,causal>+merge"}[dom_w.w["kind"]]
    peak_tc = pk["tc_sust"] or pk["tc"]
    roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": achieved, "peak": peak_tc,
                "unit": "TFLOP/s", "frac": achieved / peak_tc,
                "peak_source": f"{pk['src']} bf16 sustained (fp16 dense rate = bf16 rate)",
                "traffic": traffic_for(kernel_name)}
    extra = {}
    for w in wls:
        if w.w["kind"] == "paged":
            t = per_call[f"{w.name}:e4m3_paged_to_fp16"]
            gbs = w.bridge_bytes / (t * 1e-3) / 1e9
            t_b2b = bridge_back_to_back(torch, w)
            gbs_b2b = w.bridge_bytes / (t_b2b * 1e-3) / 1e9
            extra["bridge"] = {"achieved": gbs, "unit": "GB/s", "peak": pk["hbm"],
                               "frac": gbs / pk["hbm"], "bytes_per_launch": w.bridge_bytes,
                               "timing": "CUDA events around the call inside the step",
                               "traffic": traffic_for("e4m3_bridge_kernel"),
                               "back_to_back": {"us_per_launch": t_b2b * 1e3,
                                                "achieved": gbs_b2b,
                                                "frac": gbs_b2b / pk["hbm"],
                                                "timing": "CUDA-graph replay of 20 calls in a row"}}
    for w in wls:
        if w.w["kind"] == "vsa":
            t = per_call[f"{w.name}:vsa_select_blocks"]
            S = w.q.shape[2]
            sel_bytes = 2 * w.q.numel() * 2 + w.idx.numel() * 4   # Q and K read once, idx written
            gbs = sel_bytes / (t * 1e-3) / 1e9
            extra["select"] = {"ms": t, "achieved": gbs, "unit": "GB/s", "peak": pk["hbm"],
                               "frac": gbs / pk["hbm"], "bytes_per_call": sel_bytes,
                               "kernels": "vsa_pool_kernel + vsa_score_kernel + vsa_topk_kernel "
                                          "(+ its fallback form for rows with many undecided keys)",
                               "timing": "CUDA events around the call inside the step"}
    per_variant = {}
    for w in wls:
        t = sum(v for k, v in per_call.items() if k.startswith(w.name + ":"))
        per_variant[w.name] = {"ms": t, "tflops": w.flops / (t * 1e-3) / 1e12}

    # ---- end to end through the public API with host buffers.  Every step copies each
    # sub-workload's inputs from pinned host memory and reads its outputs back; a copy
    # stream moves data while the compute stream runs the previous sub-workload.
    e2e = None
    if not args.no_e2e:
        # Two device buffer sets per sub-workload, used on alternate steps: the
        # inputs of step s+1 are copied while step s computes on the other set, and
        # a set is refilled only after the compute two steps back has finished with
        # it and its outputs have been read back.
        sets = [wls, [Workload(n, gb, torch, dev, hosts[n]) for n in names]]
        h2d = 0
        d2h = 0
        ins, outs = {}, {}
        for p_, ws_ in enumerate(sets):
            for w in ws_:
                ins[(p_, w.name)] = []
                for dtens, i in w.h2d_pairs():
                    hp = torch.from_numpy(np.ascontiguousarray(w.host[i])).pin_memory()
                    ins[(p_, w.name)].append((hp, dtens))
                    if p_ == 0:
                        h2d += hp.numel() * hp.element_size()
                outs[(p_, w.name)] = []
                for o in w.d2h():
                    outs[(p_, w.name)].append((torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
                                               o))
                    if p_ == 0:
                        d2h += o.numel() * o.element_size()
        h2d_s = torch.cuda.Stream()     # inputs in
        d2h_s = torch.cuda.Stream()     # results out
        comp_s = stream
        ev = lambda: torch.cuda.Event()
        last_done = {}                  # (set, workload): compute that last used the set
        last_read = {}                  # (set, workload): its outputs copied back
        n_step = [0]

        def e2e_step():
            p_ = n_step[0] & 1
            n_step[0] += 1
            ready = {}
            for w in sets[p_]:                      # all input copies queue up front
                key = (p_, w.name)
                with torch.cuda.stream(h2d_s):
                    if key in last_done:
                        h2d_s.wait_event(last_done[key])   # step s-2 done with this set
                    for h, d in ins[key]:
                        d.copy_(h, non_blocking=True)
                    ready[key] = ev()
                    ready[key].record(h2d_s)
            for w in sets[p_]:
                key = (p_, w.name)
                comp_s.wait_event(ready[key])
                if key in last_read:
                    comp_s.wait_event(last_read[key])       # step s-2 outputs read back
                for _, fn in w.calls():
                    fn()
                done = ev()
                done.record(comp_s)
                last_done[key] = done
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(done)
                    for h, d in outs[key]:
                        h.copy_(d, non_blocking=True)
                    rd = ev()
                    rd.record(d2h_s)
                    last_read[key] = rd

        e2e_step()
        e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(4, 2 * (args.steps // 6))
        barrier(world, dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp_s)
        for _ in range(n_e2e):
            e2e_step()
        comp_s.wait_stream(h2d_s)
        comp_s.wait_stream(d2h_s)
        e1.record(comp_s)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        wall_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        if gb.device_status() != 0:
            raise RuntimeError("device status flags set during the end-to-end steps")
        e2e = {"value": world * flops_step / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e_ms, "wall_ms_per_step": wall_ms, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "overlap": "two device buffer sets on alternate steps; inputs copied on an H2D "
                          "stream and results on a D2H stream while the other set computes"}
        del sets[1]

    if args.small == "on" and args.workload == "all":
        for n in ("dense_small", "causal_small"):
            extra[n] = measure_small(gb, torch, dev, n, args.steps, args.warmup, pk)
    if args.decode == "on" and args.workload == "all":
        extra["decode"] = measure_decode(gb, torch, dev, args.steps, args.warmup, pk)
    if args.masked == "on" and args.workload == "all":
        extra["masked"] = measure_masked(gb, torch, dev, args.steps, args.warmup, pk)
    if args.paged_fused == "on" and args.workload == "all":
        extra["paged_fused"] = measure_paged_fused(gb, torch, dev, args.steps, args.warmup, pk)
    if args.vsa_full == "on" and args.workload == "all":
        extra["vsa_full"] = measure_vsa_full(gb, torch, dev, args.steps, args.warmup, pk)
    if args.vsa_coarse == "on" and args.workload == "all":
        extra["vsa_coarse"] = measure_vsa_coarse(gb, torch, dev, args.steps, args.warmup, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        done, secs, desc = oracle_sample(names, budget_s=args.ref_budget)
        cpu = {"value": done / secs / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": desc + f" ({secs:.1f} s of CPU time, numpy float64)"}

    if rank == 0:
        line = {"metric": "attention useful TFLOP/s", "value": value, "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                "data": "synthetic",
                "config": {"workload": "+".join(names),
                           "shapes": {n: {k: v for k, v in inputs.WORKLOADS[n].items() if k != "seed"}
                                      for n in names},
                           "parallelism": "replicas" if world > 1 else "single_gpu",
                           "l2": "inputs larger than L2 (about 1.7 GB touched per step), no flush"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clock_info, "per_call_ms": per_call, "per_call_cv": per_call_cv,
                "per_variant": per_variant}
        line.update(extra)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
