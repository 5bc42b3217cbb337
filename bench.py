"""Throughput of the routed-expert layer hot path on GB300.

One step = one forward pass of the whole layer over one batch of T tokens:
route (logits, top-K, gates, slots) -> dispatch -> grouped SwiGLU experts ->
combine, through the C ABI (`--config train` adds the combine, expert,
dispatch and router backward).  The headline workload (the default) is the
wide layer, T=32768 d=4096 N=32 K=4 h=2048, the largest configuration on one
GPU; at N=1 the OLMoE-like, fine-grained (Zipf) and training-step workloads
are measured after it, with fewer steps, under "workloads".  Inputs are
seeded synthetic tensors resident in HBM; between timed steps L2 is flushed
by writing a 512 MiB buffer (outside the per-step events).  Every step is
timed with CUDA events on the launching stream; `value` is tokens/s of the
whole job (all ranks), `e2e` the same metric through the public Python API
with the step's input copied from pinned host memory and its output read
back inside the timed region.

With --gpus N > 1 (torchrun, one process per GPU) every rank runs an
independent layer replica on its own tokens: there is no data-path collective;
a barrier brackets the timed region and the time is the max over ranks.

--impl reference times the CPU oracle on a bounded sample of the same
workload, on all host cores (tokens split for routing, dispatch and combine,
routes or experts for the expert FFN; the oracle's arithmetic is unchanged),
and prints the same line with "impl": "reference".
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer tokens/s on 1 GB300"
L2_FLUSH_BYTES = 512 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0, source="fallback")


def workload_name(cfg):
    cf = cfg.cf_num / cfg.cf_den
    s = (f"{cfg.name}: T={cfg.T} d={cfg.d} N={cfg.N} K={cfg.K} h={cfg.h} cf={cf:g} "
         f"cap={cfg.cap}")
    if cfg.zipf_s:
        s += f" zipf={cfg.zipf_s}"
    if cfg.backward:
        s += " fwd+bwd"
    return s


def algorithmic(cfg, A):
    """Bytes / FLOPs each step must move or compute (tails and re-reads excluded)."""
    T, d, K, h, N = cfg.T, cfg.d, cfg.K, cfg.h, cfg.N
    out = dict(
        route_flop=2.0 * T * N * d,
        dispatch_bytes=2.0 * T * d + 2.0 * A * d + 4.0 * T * K,
        gemm_flop=6.0 * d * h * A,
        combine_bytes=2.0 * A * d + 2.0 * T * d + 8.0 * T * K,
    )
    if cfg.backward:
        out.update(combine_bwd_bytes=2.0 * T * d + 2.0 * A * d + 2.0 * A * d + 8.0 * T * K,
                   dispatch_bwd_bytes=2.0 * A * d + 4.0 * T * d + 4.0 * T * K,
                   gemm_bwd_flop=12.0 * d * h * A,
                   # dispatch backward fused with the router's dx term and dlogit
                   dispatch_router_bwd_bytes=2.0 * A * d + 4.0 * T * d + 24.0 * T * K + 4.0 * N * d,
                   router_dw_bytes=2.0 * T * d + 8.0 * T * K + 4.0 * N * d)
    return out


def gemm_traffic(workload, kernel="grouped_gemm", sources=("grouped_gemm.cu", "moe_common.cuh")):
    """DRAM bytes per call of a GEMM from its committed ncu summary
    (profiles/<kernel>_<workload>_ncu.md), or None if there is none for this
    workload or the kernel sources have changed since the counters were taken
    (the summary names the sha256 of the sources it was captured with)."""
    import hashlib
    csrc = os.path.join(ROOT, "combine_expert_gemm_gb300", "csrc")
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_ncu.md")
    if not os.path.exists(prof):
        return None
    h = hashlib.sha256()
    for name in sources:
        h.update(open(os.path.join(csrc, name), "rb").read())
    sha = h.hexdigest()
    for line in open(prof):
        f = line.split()
        # "traffic-per-call: <bytes> bytes; kernel source sha256 <hex>"
        if len(f) >= 7 and f[0] == "traffic-per-call:" and f[6] == sha:
            return int(f[1])
    return None


def replica_config(cfg, rank):
    """The workload of one replica: rank r routes its own tokens (seed offset
    by 1000 r); rank 0 runs the named workload itself."""
    return cfg.with_(seed=cfg.seed + 1000 * rank) if rank else cfg


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself when there is one rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}




# ---------------------------------------------------------------- GPU arm --

# our kernels per step: route 6 (router-weight pack, logits, top-K, block
# ranks, scan, slot assignment), dispatch 1, experts 2, combine 1; backward:
# combine 1, experts 4 (two data-gradient and two weight-gradient GEMMs),
# dispatch + router dx 1, router dW 1 or 2 (the chunk sums need a second kernel)
FWD_LAUNCHES = 10
SIDE_WORKLOADS = ("olmoe", "fine_zipf", "train")


def launches_per_step(cfg):
    if not cfg.backward:
        return FWD_LAUNCHES
    return FWD_LAUNCHES + 6 + (2 if (cfg.T + 127) // 128 > 1 else 1)


class Layer:
    """Device inputs and buffers of one layer instance, and its step."""

    def __init__(self, moe, cfg, dev, rank=0):
        import torch
        self.moe, self.cfg, self.dev = moe, cfg, dev

        def bf(a):
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

        rcfg = replica_config(cfg, rank)
        self.x_np = synth.gen_x(rcfg)
        self.dy_np = synth.gen_dy(rcfg) if cfg.backward else None
        self.wg, self.wu, self.wd = (bf(a) for a in synth.gen_expert_weights(cfg))
        self.wr = torch.from_numpy(synth.gen_router(cfg)).to(dev)
        b_np = synth.gen_bias(cfg)
        self.bias = None if b_np is None else torch.from_numpy(b_np).to(dev)
        self.x = bf(self.x_np)
        self.dy = bf(self.dy_np) if cfg.backward else None
        self.shape = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
        self.buf = moe.LayerBuffers(self.shape, dev, save_for_backward=cfg.backward)
        self.bwd = moe.BackwardBuffers(self.shape, dev) if cfg.backward else None
        self.phases = ["route", "dispatch", "ffn", "combine"] + (
            ["combine_bwd", "ffn_bwd", "dispatch_router_bwd", "router_dw"] if cfg.backward else [])
        self.stream = torch.cuda.current_stream()

    def step(self, ev=None, split=True):
        """One layer step.  split=False records only the step's first and last
        events: events between the calls would order each call after the
        previous one has drained and hide the overlap that programmatic
        dependent launch gives a caller."""
        moe, s, b, w = self.moe, self.shape, self.buf, self.bwd
        n = len(self.phases)

        def mark(i):
            if ev is not None and (split or i == 0 or i == n):
                ev[i].record(self.stream)
        mark(0)
        moe.route(s, self.x, self.wr, self.bias, b.topk_idx, b.topk_gate, b.route_row,
                  b.expert_count, b.expert_offset, b.expert_demand, b.route_ws)
        mark(1)
        moe.dispatch(s, self.x, b.route_row, b.x_disp)
        mark(2)
        moe.expert_ffn(s, b.x_disp, b.expert_count, b.expert_offset, self.wg, self.wu, self.wd,
                       b.h_act, b.g_save, b.u_save, b.y_disp, b.ffn_ws)
        mark(3)
        moe.combine(s, b.y_disp, b.route_row, b.topk_gate, b.y)
        mark(4)
        if self.cfg.backward:
            moe.combine_backward(s, self.dy, b.y_disp, b.route_row, b.topk_gate, w.dy_disp, w.dgate)
            mark(5)
            moe.expert_ffn_backward(s, b.x_disp, b.expert_count, b.expert_offset, self.wg, self.wu,
                                    self.wd, b.g_save, b.u_save, b.h_act, w.dy_disp, w.dx_disp,
                                    w.dw_gate, w.dw_up, w.dw_down, w.ws)
            mark(6)
            moe.dispatch_router_backward(s, w.dx_disp, b.route_row, self.wr, b.topk_idx,
                                         b.topk_gate, w.dgate, w.dlogit, w.dx)
            mark(7)
            moe.router_weight_backward(s, self.x, b.topk_idx, w.dlogit, w.dw_router,
                                       None if self.bias is None else w.dbias, w.router_ws)
            mark(8)

    def check_status(self):
        moe = self.moe
        assert moe.read_device_error(self.buf.route_ws) == 0
        assert moe.read_device_error(self.buf.ffn_ws) == 0
        if self.bwd is not None:
            assert moe.read_device_error(self.bwd.ws) == 0


def time_steps(layer, flush, steps, sampler=None, dist=None):
    """Mean ms of `steps` whole steps, L2 flushed before each (outside its events)."""
    import torch
    n = len(layer.phases)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        layer.step(evs[i], split=False)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = np.array([evs[i][0].elapsed_time(evs[i][n]) for i in range(steps)])
    return float(step_ms.mean()), t_wall, clocks


def time_phases(layer, flush, steps):
    """Mean ms of each phase over `steps` further steps with an event between the calls."""
    import torch
    n = len(layer.phases)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        layer.step(sev[i])
    torch.cuda.synchronize()
    per = np.array([[sev[i][p].elapsed_time(sev[i][p + 1]) for p in range(n)] for i in range(steps)])
    return {p: float(per[:, i].mean()) for i, p in enumerate(layer.phases)}


def fp32_fma_peak_tflops(dev, sm_mhz):
    """Plain fp32 fma peak: SMs (from the device) x 128 lanes x 2 FLOP x clock."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return 2.0 * 128 * sms * sm_mhz * 1e6 / 1e12, sms


def layer_metrics(cfg, A, ph_ms, ms, world, pk, fp32_peak):
    """tokens/s and each phase against its roofline (algorithmic work, measured peaks)."""
    alg = algorithmic(cfg, A)
    gemm_tf = alg["gemm_flop"] / (ph_ms["ffn"] / 1e3) / 1e12
    dc_bytes = alg["dispatch_bytes"] + alg["combine_bytes"]
    dc_gbs = dc_bytes / ((ph_ms["dispatch"] + ph_ms["combine"]) / 1e3) / 1e9
    route_tf = alg["route_flop"] / (ph_ms["route"] / 1e3) / 1e12
    out = {
        "workload": workload_name(cfg), "tokens_per_s": world * cfg.T / (ms / 1e3),
        "ms_per_step": ms, "accepted_routes": A, "phase_ms": ph_ms,
        "gemm": {"achieved_tflops": gemm_tf, "frac": gemm_tf / pk["bf16"],
                 "frac_of_sustained": gemm_tf / pk["bf16_sus"]},
        "dispatch_combine": {"achieved": dc_gbs, "unit": "GB/s", "frac_of_measured": dc_gbs / pk["hbm"],
                             "frac_of_8tbs": dc_gbs / 8000.0,
                             "dispatch_gbs": alg["dispatch_bytes"] / (ph_ms["dispatch"] / 1e3) / 1e9,
                             "combine_gbs": alg["combine_bytes"] / (ph_ms["combine"] / 1e3) / 1e9},
        "route": {"bound": "alu", "achieved_tflops": route_tf, "peak_fp32_fma_tflops": fp32_peak,
                  "frac": route_tf / fp32_peak},
    }
    if cfg.backward:
        bt = alg["gemm_bwd_flop"] / (ph_ms["ffn_bwd"] / 1e3) / 1e12
        out["backward"] = {
            "combine_bwd_gbs": alg["combine_bwd_bytes"] / (ph_ms["combine_bwd"] / 1e3) / 1e9,
            "dispatch_router_bwd_gbs": alg["dispatch_router_bwd_bytes"] /
                                       (ph_ms["dispatch_router_bwd"] / 1e3) / 1e9,
            "router_dw_gbs": alg["router_dw_bytes"] / (ph_ms["router_dw"] / 1e3) / 1e9,
            "expert_bwd_tflops": bt, "expert_bwd_frac": bt / pk["bf16"]}
    return out


def side_workload(moe, name, dev, flush, steps, warmup, pk):
    """A shorter measurement of another workload (N=1 only): whole steps, then the phase split."""
    import torch
    cfg = synth.CONFIGS[name]
    layer = Layer(moe, cfg, dev)
    for _ in range(warmup):
        flush.zero_()
        layer.step()
    torch.cuda.synchronize()
    layer.check_status()
    ms, _, clocks = time_steps(layer, flush, steps, ClockSampler(dev.index))
    ph_ms = time_phases(layer, flush, steps)
    A = int(layer.buf.expert_offset[-1].item())
    peak, _ = fp32_fma_peak_tflops(dev, pk["sm_max_mhz"])
    out = layer_metrics(cfg, A, ph_ms, ms, 1, pk, peak)
    out.update(steps=steps, warmup=warmup, clocks=clocks,
               gpu_launches_per_step=launches_per_step(cfg),
               gemm_traffic=gemm_traffic(cfg.name))
    if cfg.zipf_s:
        out["dropped_routes"] = cfg.T * cfg.K - A
    del layer
    torch.cuda.empty_cache()
    return out


def run_ours(args, cfg, rank, world):
    import torch
    import combine_expert_gemm_gb300 as moe
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    layer = Layer(moe, cfg, dev, rank)
    shape, buf, bwd, stream = layer.shape, layer.buf, layer.bwd, layer.stream
    x, wr, bias, wg, wu, wd = layer.x, layer.wr, layer.bias, layer.wg, layer.wu, layer.wd
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        layer.step()
    torch.cuda.synchronize()
    layer.check_status()

    ms, t_wall, clocks = time_steps(layer, flush, args.steps, ClockSampler(dev.index), dist)
    ms = max_over_ranks(ms, dist, dev)
    ph_ms = time_phases(layer, flush, min(args.steps, 50))
    A = int(buf.expert_offset[-1].item())
    pk = peaks()
    fp32_peak, sms = fp32_fma_peak_tflops(dev, pk["sm_max_mhz"])
    met = layer_metrics(cfg, A, ph_ms, ms, world, pk, fp32_peak)

    # end to end: the public streamed API (combine_expert_gemm_gb300.StreamedLayer):
    # every step copies its input from pinned host memory and reads its result
    # back inside the timed region; the copies run on their own streams and
    # overlap the neighbouring steps' layer work, as a serving loop would
    x_host = torch.from_numpy(layer.x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = x.numel() * 2
    d2h = cfg.T * cfg.d * 2
    dy_host, dx_host = None, [None, None]
    if cfg.backward:
        dy_host = torch.from_numpy(layer.dy_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        dx_host = [torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d += layer.dy.numel() * 2
        d2h += cfg.T * cfg.d * 4
    sl = moe.StreamedLayer(shape, wr, bias, wg, wu, wd, dev, backward=cfg.backward)
    # warm-up: at least W steps and 0.3 s of them.  Copies to and from freshly
    # allocated pinned buffers stall once, for 20-40 ms, some 60-100 ms after
    # the allocation; a serving loop pays that once at start-up, so it stays
    # out of the timed steps
    e2e_warm = max(args.warmup, 4, int(np.ceil(300.0 / ms)))
    for i in range(e2e_warm):
        sl.submit(x_host, y_host[i % 2], dy_host, dx_host[i % 2])
    sl.synchronize()
    assert sl.status() == 0
    e2e_steps = max(10, min(args.steps, 100))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(sl.h2d)
    for i in range(e2e_steps):
        sl.submit(x_host, y_host[i % 2], dy_host, dx_host[i % 2])
    e1.record(sl.d2h)
    e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    y_e2e = y_host[(e2e_steps - 1) % 2]
    assert torch.equal(y_e2e.to(dev).view(torch.int16), buf.y.view(torch.int16)), \
        "streamed layer output differs from the timed step's"
    del sl
    torch.cuda.empty_cache()

    # dispatch fused into GEMM1 (moe_expert_ffn_gather): the same expert
    # outputs without x_disp; timed here on the same routing for comparison
    fused_ms = None
    if not cfg.backward:
        f_ms = []
        for i in range(max(5, min(args.steps, 20))):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            moe.expert_ffn_gather(shape, x, buf.route_row, buf.expert_count, buf.expert_offset, wg,
                                  wu, wd, buf.h_act, buf.g_save, buf.u_save, buf.y_disp,
                                  buf.gather_ws)
            e1.record(stream)
            e1.synchronize()
            f_ms.append(e0.elapsed_time(e1))
        assert moe.read_device_error(buf.gather_ws) == 0
        fused_ms = float(np.median(f_ms[2:]))

    # MXFP8 variant of the forward (moe_dispatch_mxfp8 -> moe_expert_ffn_mxfp8
    # -> moe_combine_mxfp8) on the same inputs and routing, timed per phase
    # outside the headline's timed region; weights are quantized once before.
    mx = None
    if not cfg.backward and cfg.d % 128 == 0 and cfg.h % 128 == 0:
        mbuf = moe.MxLayerBuffers(shape, dev)
        mw = moe.MxWeights(wg, wu, wd)

        def mx_step(ev, split):
            def mark(i):
                if split or i in (0, 4):
                    ev[i].record(stream)
            mark(0)
            moe.route(shape, x, wr, bias, mbuf.topk_idx, mbuf.topk_gate, mbuf.route_row,
                      mbuf.expert_count, mbuf.expert_offset, mbuf.expert_demand, mbuf.route_ws)
            mark(1)
            moe.dispatch_mxfp8(shape, x, mbuf.route_row, mbuf.topk_idx, mbuf.expert_count,
                               mbuf.expert_offset, mbuf.x_q, mbuf.x_sf)
            mark(2)
            moe.expert_ffn_mxfp8(shape, mbuf.x_q, mbuf.x_sf, mbuf.expert_count, mbuf.expert_offset,
                                 mw, mbuf.h_q, mbuf.h_sf, mbuf.y_q, mbuf.y_scale, mbuf.ffn_ws)
            mark(3)
            moe.combine_mxfp8(shape, mbuf.y_q, mbuf.y_scale, mbuf.route_row, mbuf.topk_gate, mbuf.y)
            mark(4)

        # whole steps without events between the calls, then the split over
        # phases from a second pass
        n_mx = max(5, min(args.steps, 20))
        mev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(2 * n_mx + 3)]
        for i in range(2 * n_mx + 3):
            flush.zero_()
            mx_step(mev[i], split=i >= n_mx + 3)
        torch.cuda.synchronize()
        assert moe.read_device_error(mbuf.ffn_ws) == 0
        mstep = np.array([mev[i][0].elapsed_time(mev[i][4]) for i in range(3, n_mx + 3)])
        mph = np.array([[mev[i][p].elapsed_time(mev[i][p + 1]) for p in range(4)]
                        for i in range(n_mx + 3, 2 * n_mx + 3)])
        mx = dict(ms=mph.mean(axis=0), step_ms=float(mstep.mean()), steps=n_mx)
        del mbuf, mw
        torch.cuda.empty_cache()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None
    alg = algorithmic(cfg, A)
    traffic = gemm_traffic(cfg.name)
    line = {
        "metric": METRIC,
        "value": world * cfg.T / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "tokens_per_gpu": cfg.T,
                   "accepted_routes": A, "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "grouped_gemm (F1 gate/up + SwiGLU, F2 down) per moe_expert_ffn call",
                     "bound": "tensor", "achieved": met["gemm"]["achieved_tflops"], "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": met["gemm"]["frac"],
                     "frac_of_sustained": met["gemm"]["frac_of_sustained"],
                     "peak_source": pk["source"] + " (burst bf16; sustained also given)",
                     "traffic": traffic},
        "dispatch_combine": met["dispatch_combine"],
        "route": dict(met["route"], sms=sms),
        "phase_ms": ph_ms,
        "phase_ms_steps": f"{min(args.steps, 50)} further steps with an event between the calls",
        "gpu_launches": launches_per_step(cfg) * args.steps,
        "e2e": {"value": world * cfg.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms, "steps": e2e_steps, "warmup": e2e_warm,
                "api": "combine_expert_gemm_gb300.StreamedLayer (layer_forward" +
                       (" + layer_backward" if cfg.backward else "") +
                       " per step; host copies overlap the neighbouring steps on their own streams)",
                "l2": "not flushed: each step's working set (weights, capacity buffers) exceeds L2"},
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if "backward" in met:
        line["backward"] = met["backward"]
    if fused_ms is not None:
        line["fused_dispatch_ffn"] = {
            "ms": fused_ms, "two_step_ms": ph_ms["dispatch"] + ph_ms["ffn"],
            "note": "moe_expert_ffn_gather (x rows gathered by cp.async inside GEMM1) vs dispatch + expert_ffn"}
    if mx is not None:
        mms = mx["ms"]
        T, d, K = cfg.T, cfg.d, cfg.K
        mx_disp_bytes = 2.0 * T * d + A * d * (1 + 1 / 32) + 8.0 * T * K
        mx_comb_bytes = A * d * (1 + 1 / 32) + 2.0 * T * d + 8.0 * T * K
        fp8_peak = 2.0 * pk["bf16"]
        mtf = alg["gemm_flop"] / (mms[2] / 1e3) / 1e12
        line["mxfp8"] = {
            "tokens_per_s": world * cfg.T / (mx["step_ms"] / 1e3),
            "ms_per_step": mx["step_ms"], "steps": mx["steps"],
            "phase_ms": {"route": float(mms[0]), "dispatch_mxfp8": float(mms[1]),
                         "ffn_mxfp8": float(mms[2]), "combine_mxfp8": float(mms[3])},
            "gemm": {"kernel": "grouped_gemm_mx_pair (F1 + SwiGLU + quantize, F2 + quantize)",
                     "bound": "tensor", "achieved": mtf, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": mtf / fp8_peak,
                     "peak_source": pk["source"] + " bf16 burst x 2 (nominal fp8 / bf16 ratio)",
                     "traffic": gemm_traffic(cfg.name, "grouped_gemm_mx",
                                             ("grouped_gemm_mx.cu", "moe_common.cuh"))},
            "dispatch_gbs": mx_disp_bytes / (mms[1] / 1e3) / 1e9,
            "combine_gbs": mx_comb_bytes / (mms[3] / 1e3) / 1e9,
            "gpu_launches_per_step": FWD_LAUNCHES,
            "note": "E4M3 data, E8M0 scales per 32; timed outside the headline region, L2 flushed"}
    del layer
    torch.cuda.empty_cache()
    if world == 1 and not args.no_side:
        side_steps = max(5, min(args.steps, 30))
        line["workloads"] = {
            n: side_workload(moe, n, dev, flush, side_steps, 3, pk)
            for n in SIDE_WORKLOADS if n != cfg.name}
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget_s)
    if dist:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------- CPU arm --

_INPUTS = {}


def _oracle_inputs(cfg):
    if cfg.name not in _INPUTS:
        _INPUTS[cfg.name] = dict(x=synth.gen_x(cfg), wr=synth.gen_router(cfg),
                                 bias=synth.gen_bias(cfg), w=synth.gen_expert_weights(cfg),
                                 dy=synth.gen_dy(cfg) if cfg.backward else None)
    return _INPUTS[cfg.name]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _ranges(n, parts):
    """`parts` contiguous ranges covering 0..n-1 (empty ones dropped)."""
    parts = max(1, min(parts, n))
    cuts = [n * i // parts for i in range(parts + 1)]
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def _expert_ranges(count, parts):
    """Contiguous expert ranges with about equal numbers of rows."""
    total = int(count.sum())
    if total == 0:
        return [(0, len(count))]
    out, start, acc = [], 0, 0
    for e, c in enumerate(count):
        acc += int(c)
        if acc * parts >= total * (len(out) + 1) and len(out) < parts - 1:
            out.append((start, e + 1))
            start = e + 1
    out.append((start, len(count)))
    return [r for r in out if r[1] > r[0]]


def oracle_layer(cfg, inp, tokens, threads):
    """The oracle on the first `tokens` tokens of the workload (capacity scaled
    to the sample): the forward, and for a training workload the combine,
    expert, dispatch and router backward.  The work is split over `threads`
    host threads -- tokens for routing, combine and the backward movements,
    routes for the expert forward, experts for the expert backward -- and
    each share runs an unchanged oracle call (ctypes releases the GIL while
    the C code runs); the token-order slot assignment and the dispatch run
    once.  Returns the outputs."""
    import oracle
    sub = cfg.with_(T=tokens)
    K, N, cap = cfg.K, cfg.N, sub.cap
    x = inp["x"][:tokens]
    wr, bias = inp["wr"], inp["bias"]
    wg, wu, wd = inp["w"]
    tr = _ranges(tokens, threads)
    with ThreadPoolExecutor(threads) as ex:
        logits = np.concatenate(list(ex.map(lambda r: oracle.router_logits(x[r[0]:r[1]], wr, bias),
                                            tr)))
        tk = list(ex.map(lambda r: oracle.topk_gates(logits[r[0]:r[1]], K), tr))
        idx = np.concatenate([a for a, _ in tk])
        gate = np.concatenate([b for _, b in tk])
        row, count, offset, demand = oracle.route_slots(idx, N, cap)
        R = min(N * cap, tokens * K)
        A = int(offset[-1])
        x_disp = oracle.dispatch(x, row, R)
        # expert forward by routes (rows 0..A-1; the expert of row r is the one
        # whose interval holds it)
        rows = np.arange(A, dtype=np.int32)
        experts = (np.searchsorted(offset, rows, side="right") - 1).astype(np.int32)
        h_act = np.zeros((R, cfg.h), np.uint16)
        y_disp = np.zeros((R, cfg.d), np.uint16)
        g_save = np.zeros((R, cfg.h), np.uint16) if cfg.backward else None
        u_save = np.zeros((R, cfg.h), np.uint16) if cfg.backward else None

        def ffn(r):
            a, b = r
            h, g, u, y = oracle.expert_ffn_rows(rows[a:b], experts[a:b], x_disp, wg, wu, wd,
                                                save=cfg.backward)
            h_act[a:b], y_disp[a:b] = h, y
            if cfg.backward:
                g_save[a:b], u_save[a:b] = g, u
        list(ex.map(ffn, _ranges(A, threads)))
        y = np.concatenate(list(ex.map(
            lambda r: oracle.combine(y_disp, row[r[0]:r[1]], gate[r[0]:r[1]]), tr)))
        out = dict(logits=logits, topk_idx=idx, topk_gate=gate, route_row=row, expert_count=count,
                   expert_offset=offset, x_disp=x_disp, h_act=h_act, y_disp=y_disp, y=y)
        if not cfg.backward:
            return out
        dy = inp["dy"][:tokens]
        dy_disp = np.zeros((R, cfg.d), np.uint16)

        def cbwd(r):
            a, b = r
            dd, dg = oracle.combine_bwd(dy[a:b], y_disp, row[a:b], gate[a:b])
            mine = row[a:b][row[a:b] >= 0]
            dy_disp[mine] = dd[mine]
            return dg
        dgate = np.concatenate(list(ex.map(cbwd, tr)))
        dx_disp = np.zeros((R, cfg.d), np.uint16)
        dwg = np.zeros(wg.shape, np.float32)
        dwu = np.zeros(wu.shape, np.float32)
        dwd = np.zeros(wd.shape, np.float32)

        def ebwd(r):
            e0, e1 = r
            dxd, g_, u_, d_ = oracle.expert_ffn_bwd(count[e0:e1], offset[e0:e1 + 1], x_disp,
                                                    g_save, u_save, h_act, dy_disp, wg[e0:e1],
                                                    wu[e0:e1], wd[e0:e1])
            a, b = int(offset[e0]), int(offset[e1])
            dx_disp[a:b] = dxd[a:b]
            dwg[e0:e1], dwu[e0:e1], dwd[e0:e1] = g_, u_, d_
        list(ex.map(ebwd, _expert_ranges(count, threads)))
        dx = np.concatenate(list(ex.map(
            lambda r: oracle.dispatch_bwd(dx_disp, row[r[0]:r[1]], r[1] - r[0]), tr)))
        rb = list(ex.map(lambda r: oracle.router_bwd(
            x[r[0]:r[1]], wr, idx[r[0]:r[1]], gate[r[0]:r[1]], dgate[r[0]:r[1]],
            dx=dx[r[0]:r[1]], with_bias=bias is not None), tr))
        out.update(dgate=dgate, dy_disp=dy_disp, dx_disp=dx_disp, dw_gate=dwg, dw_up=dwu,
                   dw_down=dwd, dlogit=np.concatenate([v[0] for v in rb]),
                   dx=np.concatenate([v[1] for v in rb]),
                   dw_router=np.sum([v[2] for v in rb], axis=0, dtype=np.float64))
        return out


def _oracle_seconds(cfg, tokens, threads):
    inp = _oracle_inputs(cfg)
    t0 = time.perf_counter()
    oracle_layer(cfg, inp, tokens, threads)
    return time.perf_counter() - t0


def _sample_tokens(cfg, seconds, threads):
    """Tokens the oracle gets through in about `seconds` on `threads` threads."""
    _oracle_inputs(cfg)  # generate the inputs outside the probe
    probe = min(cfg.T, 4 * threads)
    t = _oracle_seconds(cfg, probe, threads)
    return int(max(1, min(cfg.T, probe * seconds / max(t, 1e-3))))


def cpu_baseline(cfg, budget_s):
    """The oracle timed on one host thread and on all host cores, each on a
    bounded sample of about budget_s / 2 seconds."""
    cores = host_cores()
    what = f"oracle forward{' + backward' if cfg.backward else ''}"
    split = ("tokens split for routing, combine and the backward movements, routes for the "
             "expert forward, experts for the expert backward" if cfg.backward else
             "tokens split for routing and combine, routes for the expert forward")
    n1 = _sample_tokens(cfg, budget_s / 2, 1)
    t1 = _oracle_seconds(cfg, n1, 1)
    nc = _sample_tokens(cfg, budget_s / 2, cores)
    tc = _oracle_seconds(cfg, nc, cores)
    return {"value": nc / tc, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} on the first {nc} of {cfg.T} tokens (capacity scaled to the "
                      f"sample), {tc:.1f} s on {cores} threads: {split}",
            "single_thread": {"value": n1 / t1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{what} on the first {n1} tokens, {t1:.1f} s, 1 thread"}}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    cores = host_cores()
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    tokens = _sample_tokens(cfg, per_step, cores)
    for _ in range(args.warmup):
        _oracle_seconds(cfg, tokens, cores)
    times = [_oracle_seconds(cfg, tokens, cores) for _ in range(args.steps)]
    ms = 1e3 * float(np.mean(times))
    v = tokens / (ms / 1e3)
    sample = (f"each step: oracle forward{' + backward' if cfg.backward else ''} on the first "
              f"{tokens} of {cfg.T} tokens (capacity scaled to the sample), {cores} threads")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_name(cfg), "tokens_per_step": tokens},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="wide", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the other workloads measured after the headline at N=1")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 with torchrun")
    cfg = synth.CONFIGS[args.config]
    line = (run_reference if args.impl == "reference" else run_ours)(args, cfg, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
