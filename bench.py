"""Benchmark of the block-sparse attention backward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step = one pass of the backward hot path over one batch of synthetic input: the k2q
inversion and the backward (preprocess with the work order, main kernel, dQ postprocess), all
through the C ABI (libvsa.so).  The forward runs once before the timed region
to produce O and lse (its own time is reported under "fwd").

value   bwd TFLOPS on selected blocks: pairs x 5 x (2 x 64 x 64 x 128) flop / step time, summed
        over ranks, inputs resident in HBM (the step reads about 1 GB, far more than the 129 MB
        L2, so no separate flush), timed with CUDA events on the launching stream.
e2e     the same metric with host buffers: every step copies the inputs from pinned host memory
        to the device and the gradients back, inside the timed region.
roofline  the main kernel against the measured dense 16-bit tensor peak (MEASURED_PEAKS.json), with
          its fraction of the nominal 2.25 PFLOP/s and its ncu tensor-pipe activity beside it.
cpu_baseline  the CPU oracle timed on a bounded sample of the same workload (rank 0, N = 1).

With --impl reference the CPU oracle is the timed implementation (rank 0 only).
Multi-GPU (torchrun): every rank runs its own copy of the workload (weak scaling, independent
(b, h) problems, no data-path collective); the time is the max over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)



def flop_per_pair(blk):
    """5 GEMMs of a selected (q block, kv block) pair of `blk`-token blocks, head_dim 128."""
    return 5 * 2 * blk * blk * 128
METRIC = "bwd TFLOPS on selected blocks (5 GEMMs/pair) and % of BF16 tensor peak, 1 GB300"
# The sm_100a kernel's published TFLOPS at the same shapes (B=1, H=8, D=128, 25 % density).
PAGES_TFLOPS = {"4k_25pct": 381.0, "32k_25pct": 794.0, "131k_25pct": 736.0, "262k_25pct": 784.0,
                "524k_25pct": 771.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="32k_25pct")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def kernel_code_hash(text):
    """sha256 of a CUDA source with its comments removed and its whitespace collapsed: it changes
    when the code does, not when only comments do."""
    import hashlib
    import re
    t = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    t = re.sub(r"//[^\n]*", " ", t)
    t = re.sub(r"\s+", " ", t).strip()
    return hashlib.sha256(t.encode()).hexdigest()


def main_kernel_profile(config):
    """(DRAM bytes per main-kernel launch, tensor-pipe active fraction) from the committed ncu
    summary of this workload, or (None, None) when there is none or the kernel's code changed
    since it was captured."""
    import re
    prof = os.path.join(ROOT, "profiles", "bwd_main_%s.md" % config.split("_")[0])
    src = os.path.join(ROOT, "block_sparse_video_tok_gb300", "csrc", "bwd_main.cu")
    if not os.path.exists(prof):
        return None, None
    text = open(prof).read()
    m_code = re.search(r"code sha256 at capture: `([0-9a-f]{64})`", text)
    m_tr = re.search(r"traffic_bytes_per_launch \| (\d+)", text)
    m_tp = re.search(r"sm__pipe_tensor_cycles_active \| ([0-9.]+) %", text)
    if not (m_code and m_tr):
        return None, None
    if kernel_code_hash(open(src).read()) != m_code.group(1):
        return None, None
    return int(m_tr.group(1)), (float(m_tp.group(1)) / 100.0 if m_tp else None)


def main_kernel_traffic(config):
    """DRAM bytes per main-kernel launch from the committed ncu summary (see main_kernel_profile)."""
    return main_kernel_profile(config)[0]


# Nominal dense 16-bit tensor rate of a GB300 (PFLOP/s at its maximum clock); context only, the
# roofline's peak is the measured one.
NOMINAL_BF16_TFLOPS = 2250.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), \
            d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# ------------------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.lines = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001 - clocks are reported as unavailable
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ distributed


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist, device):
    if dist is not None:
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------ CPU oracle


class OracleSampler:
    """The CPU oracle's backward on a bounded sample of the workload: the dQ rows of the first m
    q blocks and the dK/dV rows of kv blocks 0 and 1 of one (b, h) head.  O and lse of the rows
    the sample needs come from the oracle forward, computed once (not timed)."""

    def __init__(self, case, head=(0, 0)):
        from block_sparse_video_tok_gb300 import workloads as wl
        from oracle import oracle as orc
        self.orc = orc
        b, h = self.head = head
        self.sub = {n: wl.to_f64(case[n][b:b + 1, h:h + 1]) for n in ("q", "k", "v", "do")}
        self.idx = case["q2k_idx"][b:b + 1, h:h + 1]
        self.num = case["q2k_num"][b:b + 1, h:h + 1]
        self.nb, self.vbs, self.sc = case["nb"], case["vbs"], case["sm_scale"]
        self.blk = case.get("blk", 64)
        self.k2q_idx, self.k2q_num, _ = orc.invert(self.idx, self.num, self.nb)
        S, D = self.sub["q"].shape[2:]
        self.o = np.zeros((1, 1, S, D))
        self.lse = np.zeros((1, 1, S))
        self.have = set()

    def _forward(self, blocks):
        blocks = [i for i in blocks if i not in self.have]
        if not blocks:
            return
        o, lse = self.orc.fwd(self.sub["q"], self.sub["k"], self.sub["v"], self.idx, self.num,
                              self.vbs, self.sc, blk=self.blk, qblocks=blocks)
        for i in blocks:
            r = slice(self.blk * i, self.blk * (i + 1))
            self.o[0, 0, r] = torch.from_numpy(o[0, 0, r]).to(torch.bfloat16).to(
                torch.float64).numpy()
            self.lse[0, 0, r] = lse[0, 0, r].astype(np.float32)
            self.have.add(i)

    def pairs_q(self, m):
        return int(sum(len(set(self.idx[0, 0, i, :self.num[0, 0, i]].tolist())) for i in range(m)))

    def pairs_kv(self, m):
        return int(self.k2q_num[0, 0, :m].sum())

    def run(self, m):
        """Time one sample: dQ rows of q blocks 0..m-1 and dK/dV rows of kv blocks 0..m-1.
        Returns (TFLOPS, seconds)."""
        m = max(1, min(m, self.nb))
        need = set(range(m))
        for j in range(m):
            need.update(int(i) for i in self.k2q_idx[0, 0, j, :self.k2q_num[0, 0, j]])
        self._forward(sorted(need))
        s = self.sub
        t0 = time.perf_counter()
        self.orc.bwd(s["q"], s["k"], s["v"], self.o, s["do"], self.lse, self.idx, self.num,
                     self.vbs, self.sc, blk=self.blk, qblocks=list(range(m)),
                     kvblocks=list(range(m)))
        t = time.perf_counter() - t0
        # The oracle's dQ loop recomputes S, dP and forms dQ (3 GEMM-sized products per pair);
        # its dK/dV loop recomputes S, dP and forms dV, dK (4 per pair): a pair completed = 7.
        done = (3 * self.pairs_q(m) + 4 * self.pairs_kv(m)) / 7.0
        return done * flop_per_pair(self.blk) / t / 1e12, t

    def size_for(self, target_s):
        """m whose sample takes about target_s seconds (from a small calibration run)."""
        m0 = min(max(4, 2 * self.orc.num_threads()), self.nb)  # enough blocks for every thread
        _, t = self.run(m0)
        return int(max(1, min(self.nb, m0 * target_s / max(t, 1e-3))))

    def describe(self, m):
        b, h = self.head
        return ("oracle backward (fp64, OpenMP) on head (b=%d,h=%d): dQ rows of q blocks 0..%d "
                "(%d pairs) and dK/dV rows of kv blocks 0..%d (%d pairs); TFLOPS counted as "
                "completed pairs x 5 GEMMs" % (b, h, m - 1, self.pairs_q(m), m - 1,
                                               self.pairs_kv(m)))


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from block_sparse_video_tok_gb300 import workloads as wl
    case = wl.make_config(args.config)
    sampler = OracleSampler(case)
    # Each step is a bounded sample sized so that all K + W steps take about a minute.
    per_step = min(2.0, 60.0 / max(1, args.steps + args.warmup))
    m = sampler.size_for(per_step)
    for _ in range(args.warmup):
        sampler.run(m)
    vals, secs = [], []
    for _ in range(args.steps):
        v, t = sampler.run(m)
        vals.append(v)
        secs.append(t)
    value = float(np.mean(vals))
    cores = sampler.orc.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * float(np.mean(secs)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": sampler.describe(m)},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ GPU arm


def main():
    args = parse()
    dist, rank, world, local = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return rc

    from block_sparse_video_tok_gb300 import build as vsa_build
    from block_sparse_video_tok_gb300 import vsa
    from block_sparse_video_tok_gb300 import workloads as wl
    if rank == 0:
        vsa_build.build()
    if dist is not None:
        dist.barrier()
    vsa_build.build()
    assert torch.cuda.is_available(), "the GPU arm needs CUDA"
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()

    cfg = dict(wl.CONFIGS[args.config] if args.config in wl.CONFIGS else
               wl.LONG_CONFIGS[args.config])
    case = wl.make_config(args.config, seed=cfg["seed"] + rank)
    B, H, S, nb = case["B"], case["H"], case["S"], case["nb"]
    pairs = wl.selected_pairs(case["q2k_idx"], case["q2k_num"], nb)
    dev = {n: case[n].to(device) for n in ("q", "k", "v", "do")}
    q2k_idx = torch.from_numpy(case["q2k_idx"]).to(device)
    q2k_num = torch.from_numpy(case["q2k_num"]).to(device)
    vbs = torch.from_numpy(case["vbs"]).to(device)
    sc = case["sm_scale"]

    # Forward once (operands of the backward), then time it on its own.
    fws = torch.empty(vsa.vsa_fwd_workspace_bytes(B, H, S), dtype=torch.uint8, device=device)
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device=device)
    vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], q2k_idx, q2k_num, vbs, sc, o=o, lse=lse,
                workspace=fws)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    n_fwd = 5
    for _ in range(n_fwd):
        vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], q2k_idx, q2k_num, vbs, sc, o=o, lse=lse,
                    workspace=fws)
    f1.record()
    torch.cuda.synchronize()
    fwd_ms = f0.elapsed_time(f1) / n_fwd

    k2q_idx = torch.empty((B, H, nb, nb), dtype=torch.int32, device=device)
    k2q_num = torch.empty((B, H, nb), dtype=torch.int32, device=device)
    dq, dk, dv = (torch.empty_like(dev["q"]) for _ in range(3))
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device=device)
    # invert (bitmap, compact), zeroing of the workspace header, statistics (Delta, dQ zeroing,
    # K/V to fp16, work order), convert_t (Q, dO to fp16), main, postprocess
    kernels_per_step = 7

    def step(events=None, inv=None):
        if inv is not None:
            inv[0].record()
        vsa.vsa_invert_indices(q2k_idx, q2k_num, nb, k2q_idx, k2q_num)
        if inv is not None:
            inv[1].record()
        vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num, vbs, sc,
                    dq=dq, dk=dk, dv=dv, workspace=ws, events=events)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert vsa.vsa_read_device_error(ws) == 0

    K = args.steps
    ev = [{n: torch.cuda.Event(enable_timing=True) for n in
           ("start", "before_main", "after_main", "end")} for _ in range(K)]
    inv = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in ev:   # create the CUDA events before the timed region
        for x in e.values():
            x.record()
    for a, b_ in inv:
        a.record()
        b_.record()
    torch.cuda.synchronize()

    sampler = ClockSampler(device) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier(dist, device)
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(K):
        step(ev[k], inv[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    clocks = sampler.stop() if sampler else None
    total_ms = reduce_max(dist, t_start.elapsed_time(t_end), device)
    main_ms = [e["before_main"].elapsed_time(e["after_main"]) for e in ev]
    pre_ms = [e["start"].elapsed_time(e["before_main"]) for e in ev]
    post_ms = [e["after_main"].elapsed_time(e["end"]) for e in ev]
    inv_ms = [a.elapsed_time(b_) for a, b_ in inv]
    all_pairs = reduce_sum(dist, float(pairs), device)
    fpp = flop_per_pair(case.get("blk", 64))
    value = all_pairs * fpp / (total_ms / K / 1e3) / 1e12

    # The same step captured once in a CUDA graph and replayed: one launch from the host per
    # step instead of one per kernel (the inversion and the backward enqueue only kernels on the
    # caller's stream).
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(K):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    graph_ms = reduce_max(dist, g0.elapsed_time(g1), device) / K
    assert vsa.vsa_read_device_error(ws) == 0
    del graph

    # End to end through the public API with host buffers.  Every step uploads its inputs from
    # pinned host memory and downloads its three gradients; inputs and outputs are
    # double-buffered on the device and the copies run on their own streams, so the upload of
    # step k+1 and the download of step k-1 overlap the kernels of step k.
    host_in = {n: dev[n].cpu().pin_memory() for n in ("q", "k", "v", "do")}
    host_in["o"] = o.cpu().pin_memory()
    host_in["lse"] = lse.cpu().pin_memory()
    host_in["q2k_idx"] = q2k_idx.cpu().pin_memory()
    host_in["q2k_num"] = q2k_num.cpu().pin_memory()
    host_in["vbs"] = vbs.cpu().pin_memory()
    dev_in = [{n: torch.empty_like(t, device=device) for n, t in host_in.items()}
              for _ in range(2)]
    dev_out = [[torch.empty_like(dq) for _ in range(3)] for _ in range(2)]
    host_out = [torch.empty(dq.shape, dtype=dq.dtype).pin_memory() for _ in range(3)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    s_up, s_down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {k_: [torch.cuda.Event() for _ in range(2)]
          for k_ in ("in_ready", "in_free", "out_ready", "out_free")}
    for b_ in range(2):   # all buffers start free
        ev["in_free"][b_].record(stream)
        ev["out_free"][b_].record(stream)

    def e2e_step(k_):
        b_ = k_ & 1
        di, do_ = dev_in[b_], dev_out[b_]
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev["in_free"][b_])
            for n, t in host_in.items():
                di[n].copy_(t, non_blocking=True)
            ev["in_ready"][b_].record(s_up)
        stream.wait_event(ev["in_ready"][b_])
        stream.wait_event(ev["out_free"][b_])
        vsa.vsa_invert_indices(di["q2k_idx"], di["q2k_num"], nb, k2q_idx, k2q_num)
        vsa.vsa_bwd(di["do"], di["q"], di["k"], di["v"], di["o"], di["lse"], k2q_idx, k2q_num,
                    di["vbs"], sc, dq=do_[0], dk=do_[1], dv=do_[2], workspace=ws)
        ev["in_free"][b_].record(stream)
        ev["out_ready"][b_].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev["out_ready"][b_])
            for h_, d_ in zip(host_out, do_):
                h_.copy_(d_, non_blocking=True)
            ev["out_free"][b_].record(s_down)

    for k_ in range(3):
        e2e_step(k_)
    torch.cuda.synchronize()
    # As many steps as the timed loop (at least 50), within about 3 s: the first upload and the
    # last download are not overlapped, and the steps spread them as in the device-timed loop.
    K_e2e = max(3, min(max(K, 50), int(3000.0 / max(total_ms / K, 1e-3))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    for k_ in range(K_e2e):
        e2e_step(k_)
    stream.wait_event(ev["out_free"][(K_e2e - 1) & 1])   # the last download is inside
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    e2e_ms = reduce_max(dist, e0.elapsed_time(e1), device) / K_e2e
    e2e_value = all_pairs * fpp / (e2e_ms / 1e3) / 1e12

    # A training step through the autograd binding: forward, then inversion and backward.
    from block_sparse_video_tok_gb300.autograd import block_sparse_attention
    qg, kg, vg = (dev[n].clone().requires_grad_(True) for n in ("q", "k", "v"))

    def train_step():
        for t in (qg, kg, vg):
            t.grad = None
        block_sparse_attention(qg, kg, vg, q2k_idx, q2k_num, vbs, sc).backward(dev["do"])

    for _ in range(3):
        train_step()
    torch.cuda.synchronize()
    K_train = max(3, min(K, 20))
    t0_, t1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    t0_.record(stream)
    for _ in range(K_train):
        train_step()
    t1_.record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    train_ms = reduce_max(dist, t0_.elapsed_time(t1_), device) / K_train
    train_tflops = all_pairs * fpp * 7 / 5 / (train_ms / 1e3) / 1e12

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_sus, hbm, peak_src = peaks()
    main_avg = float(np.mean(main_ms))
    achieved = pairs * fpp / (main_avg / 1e3) / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(case)
        m = sampler.size_for(12.0)
        v, t = sampler.run(m)
        cpu = {"value": v, "unit": "TFLOPS", "cores": sampler.orc.num_threads(), "kind": "oracle",
               "sample": sampler.describe(m), "seconds": t}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / PAGES_TFLOPS[args.config]) if args.config in PAGES_TFLOPS else None,
        "dtype": "f16 tensor-core operands, f32 accumulate (bf16 in/out)", "data": "synthetic",
        "config": {"workload": args.config, "B": B, "H": H, "S": S, "D": 128, "nb": nb,
                   "topk": cfg["topk"], "selection": cfg["select"], "vbs": cfg["vbs"],
                   "pairs_per_gpu": pairs, "l2": "inputs larger than L2 (no flush)",
                   "step": "invert + backward (preprocess with the work order, main, postprocess)",
                   "parallelism": "replicas over (b,h) problems, one per GPU"},
        "pct_of_peak": 100.0 * value / peak / world,
        "breakdown_ms": {"invert": float(np.mean(inv_ms)), "preprocess": float(np.mean(pre_ms)),
                         "main": main_avg, "postprocess": float(np.mean(post_ms))},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": main_kernel_profile(args.config)[0],
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "tensor_pipe_active_ncu": main_kernel_profile(args.config)[1],
                     "peak_source": "%s bf16_tflops (burst); fp16 dense rate = bf16" % peak_src,
                     "frac_of_sustained": achieved / peak_sus},
        "graph_step": {"ms": graph_ms, "tflops": all_pairs * fpp / (graph_ms / 1e3) / 1e12,
                       "note": "the same step (inversion + backward) captured in one CUDA graph "
                               "and replayed; not the headline value"},
        "fwd": {"ms": fwd_ms, "note": "operand producer, timed alone; not in the step"},
        "train_step": {"ms": train_ms, "tflops": train_tflops, "steps": K_train,
                       "note": "forward + inversion + backward through the autograd binding; "
                               "2 + 5 GEMMs per selected pair"},
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": K_e2e,
                "copies": "every step uploads its inputs and downloads dQ, dK, dV; double "
                          "buffers on copy streams overlap them with the neighbouring steps"},
        "gpu_launches": kernels_per_step * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
