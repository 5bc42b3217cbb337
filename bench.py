"""Throughput of the routed-expert layer hot path on GB300.

One step = one forward pass of the whole layer over one batch of T tokens:
route (logits, top-K, gates, slots) -> dispatch -> grouped SwiGLU experts ->
combine, through the C ABI (`--config train` adds the combine, expert,
dispatch and router backward).  Inputs are seeded synthetic tensors resident
in HBM; between timed steps L2 is flushed by writing a 512 MiB buffer (outside the
per-step events).  Every step is timed with CUDA events on the launching
stream; `value` is tokens/s of the whole job (all ranks), `e2e` the same metric
through the public Python API with the step's input copied from pinned host
memory and its output read back inside the timed region.

With --gpus N > 1 (torchrun, one process per GPU) every rank runs an
independent layer replica on its own tokens: there is no data-path collective;
a barrier brackets the timed region and the time is the max over ranks.

--impl reference times the CPU oracle (single thread) on a bounded sample of
the same workload and prints the same line with "impl": "reference".
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

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

def run_ours(args, cfg, rank, world):
    import torch
    import combine_expert_gemm_gb300 as moe

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    rcfg = replica_config(cfg, rank)
    x_np = synth.gen_x(rcfg)
    wg, wu, wd = (bf(a) for a in synth.gen_expert_weights(cfg))
    wr = torch.from_numpy(synth.gen_router(cfg)).to(dev)
    b_np = synth.gen_bias(cfg)
    bias = None if b_np is None else torch.from_numpy(b_np).to(dev)
    x = bf(x_np)
    dy = bf(synth.gen_dy(rcfg)) if cfg.backward else None
    shape = moe.Shape(cfg.T, cfg.d, cfg.N, cfg.K, cfg.h, cfg.cap)
    buf = moe.LayerBuffers(shape, dev, save_for_backward=cfg.backward)
    bwd = moe.BackwardBuffers(shape, dev) if cfg.backward else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    phases = ["route", "dispatch", "ffn", "combine"] + (
        ["combine_bwd", "ffn_bwd", "dispatch_router_bwd", "router_dw"] if cfg.backward else [])
    # our kernels per step: route 5 (logit blocks, top-K, block ranks, scan,
    # slot assignment), dispatch 1, experts 2, combine 1; backward: combine 1,
    # experts 4 (two data-gradient and two weight-gradient GEMMs), dispatch +
    # router dx 1, router dW 1 or 2 (the chunk sums need a second kernel)
    router_dw_launches = 2 if (cfg.T + 127) // 128 > 1 else 1
    launches_per_step = 9 + (6 + router_dw_launches if cfg.backward else 0)
    db = None if (bias is None or bwd is None) else bwd.dbias

    # split=False records only the step's first and last events: events between
    # the calls would order each call after the previous one has drained and
    # hide the overlap that programmatic dependent launch gives a caller
    def step(ev=None, split=True):
        def mark(i):
            if ev is not None and (split or i == 0 or i == len(phases)):
                ev[i].record(stream)
        mark(0)
        moe.route(shape, x, wr, bias, buf.topk_idx, buf.topk_gate, buf.route_row,
                  buf.expert_count, buf.expert_offset, buf.expert_demand, buf.route_ws)
        mark(1)
        moe.dispatch(shape, x, buf.route_row, buf.x_disp)
        mark(2)
        moe.expert_ffn(shape, buf.x_disp, buf.expert_count, buf.expert_offset, wg, wu, wd,
                       buf.h_act, buf.g_save, buf.u_save, buf.y_disp, buf.ffn_ws)
        mark(3)
        moe.combine(shape, buf.y_disp, buf.route_row, buf.topk_gate, buf.y)
        mark(4)
        if cfg.backward:
            moe.combine_backward(shape, dy, buf.y_disp, buf.route_row, buf.topk_gate,
                                 bwd.dy_disp, bwd.dgate)
            mark(5)
            moe.expert_ffn_backward(shape, buf.x_disp, buf.expert_count, buf.expert_offset, wg, wu,
                                    wd, buf.g_save, buf.u_save, buf.h_act, bwd.dy_disp,
                                    bwd.dx_disp, bwd.dw_gate, bwd.dw_up, bwd.dw_down, bwd.ws)
            mark(6)
            moe.dispatch_router_backward(shape, bwd.dx_disp, buf.route_row, wr, buf.topk_idx,
                                         buf.topk_gate, bwd.dgate, bwd.dlogit, bwd.dx)
            mark(7)
            moe.router_weight_backward(shape, x, buf.topk_idx, bwd.dlogit, bwd.dw_router, db,
                                       bwd.router_ws)
            mark(8)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert moe.read_device_error(buf.route_ws) == 0 and moe.read_device_error(buf.ffn_ws) == 0
    if bwd is not None:
        assert moe.read_device_error(bwd.ws) == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
           for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(evs[i], split=False)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = np.array([evs[i][0].elapsed_time(evs[i][len(phases)]) for i in range(args.steps)])
    ms = max_over_ranks(float(step_ms.mean()), dist, dev)
    # the split over phases, from a separate pass with an event between calls
    n_split = min(args.steps, 50)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
           for _ in range(n_split)]
    for i in range(n_split):
        flush.zero_()
        step(sev[i])
    torch.cuda.synchronize()
    per_phase = np.array([[sev[i][p].elapsed_time(sev[i][p + 1]) for p in range(len(phases))]
                          for i in range(n_split)])  # ms
    A = int(buf.expert_offset[-1].item())
    alg = algorithmic(cfg, A)
    pk = peaks()
    ph_ms = {p: float(per_phase[:, i].mean()) for i, p in enumerate(phases)}

    # end to end: the public streamed API (combine_expert_gemm_gb300.StreamedLayer):
    # every step copies its input from pinned host memory and reads its result
    # back inside the timed region; the copies run on their own streams and
    # overlap the neighbouring steps' layer work, as a serving loop would
    x_host = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = x.numel() * 2
    d2h = cfg.T * cfg.d * 2
    dy_host, dx_host = None, [None, None]
    if cfg.backward:
        dy_host = torch.from_numpy(synth.gen_dy(rcfg).view(np.int16)).view(torch.bfloat16).pin_memory()
        dx_host = [torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d += dy.numel() * 2
        d2h += cfg.T * cfg.d * 4
    sl = moe.StreamedLayer(shape, wr, bias, wg, wu, wd, dev, backward=cfg.backward)
    for i in range(4):
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

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return None
    gemm_s = ph_ms["ffn"] / 1e3
    dc_bytes = alg["dispatch_bytes"] + alg["combine_bytes"]
    dc_s = (ph_ms["dispatch"] + ph_ms["combine"]) / 1e3
    achieved_tf = alg["gemm_flop"] / gemm_s / 1e12
    traffic = gemm_traffic(cfg.name)
    sm_clock = clocks["sm_mhz"] if clocks else pk["sm_max_mhz"]
    fp32_peak = 2.0 * 128 * 152 * pk["sm_max_mhz"] * 1e6 / 1e12
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
                     "bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16"],
                     "frac_of_sustained": achieved_tf / pk["bf16_sus"],
                     "peak_source": pk["source"] + " (burst bf16; sustained also given)",
                     "traffic": traffic},
        "dispatch_combine": {"achieved": dc_bytes / dc_s / 1e9, "unit": "GB/s",
                             "frac_of_measured": dc_bytes / dc_s / 1e9 / pk["hbm"],
                             "frac_of_8tbs": dc_bytes / dc_s / 1e9 / 8000.0,
                             "dispatch_gbs": alg["dispatch_bytes"] / (ph_ms["dispatch"] / 1e3) / 1e9,
                             "combine_gbs": alg["combine_bytes"] / (ph_ms["combine"] / 1e3) / 1e9},
        "route": {"bound": "alu", "achieved_tflops": alg["route_flop"] / (ph_ms["route"] / 1e3) / 1e12,
                  "peak_fp32_fma_tflops": fp32_peak,
                  "frac": alg["route_flop"] / (ph_ms["route"] / 1e3) / 1e12 / fp32_peak},
        "phase_ms": ph_ms,
        "phase_ms_steps": f"{n_split} further steps with an event between the calls",
        "gpu_launches": launches_per_step * args.steps,
        "e2e": {"value": world * cfg.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "api": "combine_expert_gemm_gb300.StreamedLayer (layer_forward" +
                       (" + layer_backward" if cfg.backward else "") +
                       " per step; host copies overlap the neighbouring steps on their own streams)",
                "l2": "not flushed: each step's working set (weights 805 MB) exceeds L2"},
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if fused_ms is not None:
        line["fused_dispatch_ffn"] = {
            "ms": fused_ms, "two_step_ms": ph_ms["dispatch"] + ph_ms["ffn"],
            "note": "moe_expert_ffn_gather (x rows fetched by TMA gather4 in GEMM1) vs dispatch + expert_ffn"}
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
            "gpu_launches_per_step": 9,
            "note": "E4M3 data, E8M0 scales per 32; timed outside the headline region, L2 flushed"}
    if cfg.backward:
        bt = alg["gemm_bwd_flop"] / (ph_ms["ffn_bwd"] / 1e3) / 1e12
        line["backward"] = {
            "combine_bwd_gbs": alg["combine_bwd_bytes"] / (ph_ms["combine_bwd"] / 1e3) / 1e9,
            "dispatch_router_bwd_gbs": alg["dispatch_router_bwd_bytes"] /
                                       (ph_ms["dispatch_router_bwd"] / 1e3) / 1e9,
            "router_dw_gbs": alg["router_dw_bytes"] / (ph_ms["router_dw"] / 1e3) / 1e9,
            "expert_bwd_tflops": bt, "expert_bwd_frac": bt / pk["bf16"]}
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


def _oracle_sample(cfg, tokens):
    """Seconds the oracle takes for the forward (and, for train, the combine and
    dispatch backward) of the first `tokens` tokens of the workload."""
    import oracle
    inp = _oracle_inputs(cfg)
    sub = cfg.with_(T=tokens)
    x = inp["x"][:tokens]
    wg, wu, wd = inp["w"]
    t0 = time.perf_counter()
    out = oracle.layer_forward(x, inp["wr"], inp["bias"], wg, wu, wd, cfg.K, sub.cap,
                               save=cfg.backward)
    if cfg.backward:
        dyd, dg = oracle.combine_bwd(inp["dy"][:tokens], out["y_disp"], out["route_row"],
                                     out["topk_gate"])
        dxd, dwg, dwu, dwd = oracle.expert_ffn_bwd(out["expert_count"], out["expert_offset"],
                                                   out["x_disp"], out["g_save"], out["u_save"],
                                                   out["h_act"], dyd, wg, wu, wd)
        dx = oracle.dispatch_bwd(dxd, out["route_row"], tokens)
        oracle.router_bwd(x, inp["wr"], out["topk_idx"], out["topk_gate"], dg, dx=dx,
                          with_bias=inp["bias"] is not None)
    return time.perf_counter() - t0


def cpu_baseline(cfg, budget_s):
    t1 = _oracle_sample(cfg, 1)
    tokens = int(max(1, min(cfg.T, budget_s / max(t1, 1e-3))))
    dt = _oracle_sample(cfg, tokens)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle forward{'+backward' if cfg.backward else ''} on the first {tokens} "
                      f"of {cfg.T} tokens (capacity scaled to the sample), {dt:.1f} s, 1 thread"}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    t1 = _oracle_sample(cfg, 1)
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    tokens = int(max(1, min(cfg.T, per_step / max(t1, 1e-3))))
    for _ in range(args.warmup):
        _oracle_sample(cfg, tokens)
    times = [_oracle_sample(cfg, tokens) for _ in range(args.steps)]
    ms = 1e3 * float(np.mean(times))
    v = tokens / (ms / 1e3)
    sample = (f"each step: oracle forward{'+backward' if cfg.backward else ''} on the first "
              f"{tokens} of {cfg.T} tokens, 1 thread")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_name(cfg), "tokens_per_step": tokens},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="olmoe", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
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
