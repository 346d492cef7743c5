#!/usr/bin/env python3
"""Benchmark of the activation-sparse gated FFN on one or more GB300s.

Default workload (N=1): Llama-2-7B-shaped ReGLU FFN decode (d_model 4096,
d_ff 11008, bf16 weights, fp32 accumulation, exact gating, batch 1 token per
call), 1024 tokens per step rotating over 8 independent layer copies (2.2 GB of
weights, far larger than L2, so no L2 flush is needed).  A step is one CUDA
graph of 1024 sffn_decode calls (one kernel each at this shape).

Prints one JSON line (rank 0).  `value` is decode microseconds per token over
all ranks' tokens (lower is better).  The `prefill` object adds the second half
of the metric: token-selective prefill (L 16384, d_model 5120, d_ff 25600,
SwiGLU bf16) tokens/s for mass_thresh 0.2 / 0.5 / 0.7 / 1.0 and the tensor
roofline of its FFN GEMMs.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the decode workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-FFN µs/token & HBM GB/s vs active fraction; sparse-prefill tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained") or bf
            if hbm:
                return float(hbm), float(bf or FALLBACK_BF16_TFLOPS), float(bfs or FALLBACK_BF16_TFLOPS), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1] and parts[1] not in self.uuid:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][3]) if rows[0][3].replace(".", "").isdigit() else None,
                "samples": len(rows), "reasons": sorted(reasons)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, dist, device):
    """Element-wise maximum of this rank's timings (ms) over all ranks: the job
    takes as long as its slowest replica.  Identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def per_token_us(ms_max, steps, tokens_per_step, world):
    """Whole-job microseconds per token: the slowest replica's time over the
    tokens all replicas processed (weak scaling: each replica runs its own)."""
    return ms_max * 1e3 / (steps * tokens_per_step * world)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__ as G
    G.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    from activation_sparse_ffn_gemv_gb300 import workloads as W

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    cfg = W.CONFIGS[2]
    d, F, nlayers, T = cfg["d_model"], cfg["d_ff"], cfg["layers"], args.tokens
    dev = torch.device("cuda", local)
    layers = [W.make_ffn_layer(2, seed=1000 * rank, layer=l, device=dev) for l in range(nlayers)]
    ws_list = [sffn.Weights(L) for L in layers]
    x = W.make_tokens(2, T, seed=rank, device=dev)
    out = torch.empty_like(x)
    idx = torch.empty((T, F), dtype=torch.int32, device=dev)
    nact = torch.empty(T, dtype=torch.int32, device=dev)
    work = sffn.alloc_workspace(sffn.WS_DECODE, 1, ws_list[0], dev)
    stream = torch.cuda.Stream(device=dev)
    # the inputs and the zero-filled workspace are made on the default stream:
    # they must be complete before the decode stream uses them
    torch.cuda.synchronize()

    def enqueue(xin, oo):
        for t in range(T):
            sffn.decode(xin[t:t + 1], ws_list[t % nlayers], sffn.MODE_EXACT, out=oo[t:t + 1],
                        active_idx=idx[t:t + 1], n_active=nact[t:t + 1], workspace=work, stream=stream)

    with torch.cuda.stream(stream):
        enqueue(x, out)                      # eager warm-up: sets kernel attributes before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        enqueue(x, out)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop() if clocks else None
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks([ms], dist, dev)[0]

    # end to end: host buffers in, host buffers out, copies inside the timed region
    xh = x.cpu().pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    nh = torch.empty(T, dtype=torch.int32).pin_memory()
    xd = torch.empty_like(x)
    od = torch.empty_like(out)
    graph_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        enqueue(xd.copy_(xh), od)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph_e2e, stream=stream):
        enqueue(xd, od)
    with torch.cuda.stream(stream):
        for _ in range(2):
            xd.copy_(xh, non_blocking=True)
            graph_e2e.replay()
            outh.copy_(od, non_blocking=True)
            nh.copy_(nact, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(args.steps):
            xd.copy_(xh, non_blocking=True)
            graph_e2e.replay()
            outh.copy_(od, non_blocking=True)
            nh.copy_(nact, non_blocking=True)
        f1.record(stream)
    f1.synchronize()
    ms_e2e = max_over_ranks([f0.elapsed_time(f1)], dist, dev)[0]

    # active fraction and algorithmic bytes per token
    n_np = nact.cpu().numpy().astype(np.float64)
    a = float(n_np.mean() / F)
    r = 2.0 * d
    bytes_tok = (F * r + 2.0 * n_np.mean() * r      # gate rows + active up rows + active down rows
                 + 4.0 * F                            # gate bias
                 + 2.0 * d + 2.0 * d                  # x in, out
                 + 4.0 * n_np.mean() + 4.0)           # active index list + count
    us_tok = ms_max * 1e3 / (args.steps * T)
    total_tokens = args.steps * T * world
    value = per_token_us(ms_max, args.steps, T, world)
    hbm, bf16_peak, bf16_sus, peak_src = peaks()
    achieved = bytes_tok / (us_tok * 1e-6) / 1e9
    # one fused kernel per call when every gate chunk's CTA is resident (the
    # decode plan: C = ceil(F / R) chunks, R = ceil(F / min(#SMs, 256)) <= 256),
    # else the gate kernel and the reduction
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    R = min(256, -(-F // min(sms, 256, F)))
    kernels_per_call = 1 if -(-F // R) <= sms else 2
    res = None
    if rank == 0:
        res = {
            "metric": METRIC, "value": round(value, 4), "unit": "us/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1/d_in) weights, gate bias N(-1.2,0.3), x N(0,1)",
            "config": {"workload": "llama2-7b-reglu-decode: d_model 4096, d_ff 11008, bf16, exact gating, "
                                   "batch 1, 1024 tokens/step over 8 layer copies",
                       "d_model": d, "d_ff": F, "batch": 1, "tokens_per_step": T, "layer_copies": nlayers,
                       "mode": "exact", "l2": "inputs larger than L2: 2.2 GB of weights rotated, no flush",
                       "parallelism": f"replicas x{world}"},
            "active_fraction": round(a, 5),
            "gbps": round(achieved, 1),
            "roofline": {"bound": "hbm", "kernel": "sffn_decode call (one kernel: gate stream, active up/down rows, grid-barrier reduction)",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                         "bytes_per_launch": round(bytes_tok), "traffic": traffic_for("decode_exact_llama")},
            "e2e": {"value": round(per_token_us(ms_e2e, args.steps, T, world), 4), "unit": "us/token",
                    "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
                    "d2h_bytes_per_step": int(outh.numel() * outh.element_size() + nh.numel() * 4),
                    "copied": "x in; out and n_active back; the active_idx lists stay on the device"},
            "gpu_launches": int(args.steps * T * kernels_per_call),
            "clocks": clk,
        }
    # CPU baseline: the oracle on a bounded sample of the same workload
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(layers[0], x[: args.cpu_tokens].cpu())
    del graph, graph_e2e, layers, ws_list, idx, work
    torch.cuda.empty_cache()
    if not args.no_prefill:
        pf = bench_prefill(args, dev, rank, world, dist)
        if rank == 0:
            res["prefill"] = pf
            res["prefill_stack"] = bench_prefill_stack(args, dev)
            res["moe"] = bench_moe(args, dev)
    if not args.no_sweeps:
        sw = bench_decode_sweeps(args, dev)
        if rank == 0:
            res["decode_configs"] = sw
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return res


def run_prefill_only(args):
    import torch

    import __graft_entry__ as G
    G.build()
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    res = bench_prefill(args, torch.device("cuda", local), rank, 1, None)
    if rank != 0:
        return None
    return {"prefill": res, "prefill_stack": bench_prefill_stack(args, torch.device("cuda", local)),
            "moe": bench_moe(args, torch.device("cuda", local))}


def _time_graph(enqueue, stream, steps, warmup):
    """Capture enqueue() in a CUDA graph; device ms per replay."""
    import torch
    with torch.cuda.stream(stream):
        enqueue()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def bench_decode_sweeps(args, dev, T=256):
    """The other decode workloads.  Each point is a CUDA graph of T decode calls
    rotating over the workload's layers (far more weight bytes than L2):
    the int4 active-fraction sweep against the dense layer (speed-ups and the
    breakeven active fraction), batched tokens on the Llama shape, keep-ratio
    tiers (both scores) and the tiny fp32 layer.  Each point reports microseconds
    per token and its HBM roofline fraction on the bytes the call must read."""
    import numpy as np
    import torch

    from activation_sparse_ffn_gemv_gb300 import sffn
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    stream = torch.cuda.Stream(device=dev)
    hbm = peaks()[0]
    out = {}
    legs = set(args.sweep.split(",")) if getattr(args, "sweep", None) else None

    def want(name):
        return legs is None or name in legs

    def rowb(c):
        d = c["d_model"]
        return {"f32": 4.0 * d, "bf16": 2.0 * d, "int4_g64": d / 2 + 2.0 * d / 64}[c["wdtype"]]

    def point(us, nbytes, **kw):
        gbps = nbytes / (us * 1e-6) / 1e9
        return dict(us_per_token=round(us, 3), gbps=round(gbps, 1), frac_hbm=round(gbps / hbm, 4), **kw)

    def setup(cfgn, nl, B=1, norms=True):
        layers = [W.make_ffn_layer(cfgn, seed=100, layer=l, device=dev) for l in range(nl)]
        ws = [sffn.Weights(L) for L in layers]
        if norms:
            for w in ws:
                w.set_down_norms(sffn.down_norms(w))
        x = W.make_tokens(cfgn, T * B, seed=5, device=dev)
        F = ws[0].d_ff
        bufs = dict(o=torch.empty_like(x), idx=torch.empty((T * B, F), dtype=torch.int32, device=dev),
                    n=torch.empty(T * B, dtype=torch.int32, device=dev),
                    work=sffn.alloc_workspace(sffn.WS_DECODE, B, ws[0], dev))
        torch.cuda.synchronize()  # made on the default stream, used on `stream`
        return layers, ws, x, bufs

    def run_sparse(ws, x, bufs, B, mode, score, params):
        nl = len(ws)

        def enq():
            for t in range(T):
                sl = slice(t * B, (t + 1) * B)
                sffn.decode(x[sl], ws[t % nl], mode, score, params[t % nl], out=bufs["o"][sl],
                            active_idx=bufs["idx"][sl], n_active=bufs["n"][sl], workspace=bufs["work"],
                            stream=stream)
        return _time_graph(enq, stream, max(3, args.steps // 3), args.warmup) * 1e3 / T

    def run_dense(ws, x, bufs, B):
        nl = len(ws)

        def enq():
            for t in range(T):
                sl = slice(t * B, (t + 1) * B)
                sffn.decode_dense(x[sl], ws[t % nl], out=bufs["o"][sl], workspace=bufs["work"], stream=stream)
        return _time_graph(enq, stream, max(3, args.steps // 3), args.warmup) * 1e3 / T

    if want("int4"):
        # ---- int4 sweep: threshold tau_a = (1 - a) quantile of the layer's gate scores
        c = W.CONFIGS[4]
        nl = c["layers"]
        layers, ws, x, bufs = setup(4, nl)
        calib = W.make_tokens(4, 256, seed=77, device=dev)
        sc_ws = sffn.alloc_workspace(sffn.WS_DECODE, 8, ws[0], dev)
        torch.cuda.synchronize()
        taus = []
        for w in ws:
            sc = torch.cat([sffn.gate_scores(calib[i:i + 8], w, sffn.SCORE_GATE, workspace=sc_ws)
                            for i in range(0, 256, 8)])
            taus.append(torch.quantile(sc.flatten()[::4].float(),
                                       torch.tensor([1.0 - a for a in c["sweep_a"]], device=dev)).tolist())
        F, r = c["d_ff"], rowb(c)
        dense_us = run_dense(ws, x, bufs, 1)
        sweep = []
        for i, a_t in enumerate(c["sweep_a"]):
            us = run_sparse(ws, x, bufs, 1, sffn.MODE_THRESHOLD, sffn.SCORE_GATE,
                            [taus[l][i] if a_t < 1.0 else 0.0 for l in range(nl)])
            a = float(bufs["n"].float().mean().item()) / F
            sweep.append(point(us, F * r * (1 + 2 * a), a_target=a_t, a=round(a, 4),
                               speedup_vs_dense=round(dense_us / us, 3)))
        # breakeven: where the sparse call takes as long as the dense layer, linear
        # between swept points ("<" / ">" outside the sweep)
        be = None
        for p0, p1 in zip(sweep, sweep[1:]):
            if p0["us_per_token"] <= dense_us <= p1["us_per_token"] and p1["us_per_token"] > p0["us_per_token"]:
                be = round(p0["a"] + (dense_us - p0["us_per_token"]) * (p1["a"] - p0["a"]) /
                           (p1["us_per_token"] - p0["us_per_token"]), 3)
                break
        if be is None and sweep:
            be = f"< {sweep[0]['a']}" if sweep[0]["us_per_token"] > dense_us else (
                f">= {sweep[-1]['a']}" if sweep[-1]["us_per_token"] <= dense_us else None)
        out["int4_threshold_sweep"] = {
            "workload": "qwen2.5-3b-swiglu-int4g64: d_model 2048, d_ff 11008, 36 layers, threshold on "
                        "|SiLU(g)|*||W_down[:,j]||, B=1",
            "dense": point(dense_us, 3 * F * r, kernel="sffn_decode_dense: every neuron, the three matrices read once"),
            "points": sweep, "breakeven_active_fraction": be}
        # int4 keep-ratio tiers (gate-and-up score: W_up read in full)
        kr4 = {}
        for M in (2, 4, 8):
            us = run_sparse(ws, x, bufs, 1, sffn.MODE_KEEP_RATIO, sffn.SCORE_GATE_UP, [1.0 / M] * nl)
            a = float(bufs["n"].float().mean().item()) / F
            kr4[str(M)] = point(us, F * r * (2 + a), a=round(a, 4), speedup_vs_dense=round(dense_us / us, 3))
        out["int4_keep_ratio"] = {"workload": "as int4_threshold_sweep, keep the top d_ff/M gate-and-up scores",
                                  "by_M": kr4}
        del layers, ws, x, bufs, sc_ws
        torch.cuda.empty_cache()

    if want("batch"):
        # ---- Llama shape, exact gating: batched tokens (the union of the tokens'
        # active rows is read once) and the dense layer at B = 1
        c = W.CONFIGS[2]
        F, r = c["d_ff"], rowb(c)
        bt = {}
        for B in (1, 2, 4, 8):
            layers, ws, x, bufs = setup(2, 8, B=B, norms=False)
            us = run_sparse(ws, x, bufs, B, sffn.MODE_EXACT, sffn.SCORE_GATE, [0.0] * 8) / B
            n = bufs["n"].cpu().numpy()
            idx = bufs["idx"].cpu().numpy()
            uni = np.mean([np.unique(np.concatenate([idx[t * B + b, : n[t * B + b]] for b in range(B)])).size
                           for t in range(T)]) / F
            bt[str(B)] = point(us, F * r * (1 + 2 * uni) / B, a_per_token=round(float(n.mean()) / F, 4),
                               union_fraction=round(float(uni), 4))
            if B == 1:
                dus = run_dense(ws, x, bufs, 1)
                bt["dense_B1"] = point(dus, 3 * F * r, speedup_of_sparse_B1=round(dus / us, 3))
            del layers, ws, x, bufs
            torch.cuda.empty_cache()
        out["llama_exact_by_batch"] = bt

    if want("keep_ratio"):
        # ---- keep-ratio tiers: the gate-and-up score (W_up read in full, only W_down
        # sparse) and the gate score (W_up and W_down sparse)
        c = W.CONFIGS[3]
        F, r = c["d_ff"], rowb(c)
        layers, ws, x, bufs = setup(3, c["layers"])
        kr = {}
        for name, score in (("gate_up", sffn.SCORE_GATE_UP), ("gate", sffn.SCORE_GATE)):
            by = {}
            for M in c["keep_M"]:
                us = run_sparse(ws, x, bufs, 1, sffn.MODE_KEEP_RATIO, score, [1.0 / M] * c["layers"])
                a = float(bufs["n"].float().mean().item()) / F
                by[str(M)] = point(us, F * r * ((2 + a) if score == sffn.SCORE_GATE_UP else (1 + 2 * a)), a=round(a, 4))
            kr[name] = by
        out["keep_ratio"] = {"workload": "qwen2.5-3b-swiglu: d_model 2048, d_ff 11008 bf16, 36 layers, keep the "
                                         "top d_ff/M scores, B=1", "by_score": kr}

        # ---- tier tables (sffn_decode_tiered): per layer a core of half the tier
        # from 64 calibration tokens (sffn_tier_core_set), the rest chosen online
        xc = W.make_tokens(3, 64, seed=99, device=dev)
        tiers = {}
        for name, score in (("gate_up", sffn.SCORE_GATE_UP), ("gate", sffn.SCORE_GATE)):
            by = {}
            for M in (4, 8):
                k = max(1, int(F / M))
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                cores = []
                for l, w in enumerate(ws):
                    sc = torch.cat([sffn.gate_scores(xc[i:i + 8], w, score) for i in range(0, 64, 8)])
                    if l == 0:
                        t0.record()
                    cores.append(sffn.tier_core_set(sc, k, k // 2))
                    if l == 0:
                        t1.record()
                torch.cuda.synchronize()

                def enq():
                    for t in range(T):
                        sffn.decode_tiered(x[t:t + 1], ws[t % c["layers"]], score, 1.0 / M, cores[t % c["layers"]],
                                           out=bufs["o"][t:t + 1], active_idx=bufs["idx"][t:t + 1],
                                           n_active=bufs["n"][t:t + 1], workspace=bufs["work"], stream=stream)
                us = _time_graph(enq, stream, max(3, args.steps // 3), args.warmup) * 1e3 / T
                a = float(bufs["n"][:T].float().mean().item()) / F
                nb = F * r * ((2 + a) if score == sffn.SCORE_GATE_UP else (1 + 2 * a))
                by[str(M)] = point(us, nb, a=round(a, 4), core=k // 2,
                                   speedup_vs_keep_ratio=round(kr[name][str(M)]["us_per_token"] / us, 3),
                                   core_set_ms=round(t0.elapsed_time(t1), 4))
            tiers[name] = by
        out["tiered"] = {"workload": "as keep_ratio, with a per-layer core of k/2 columns from 64 calibration tokens; "
                                     "core_set_ms: sffn_tier_core_set for one layer (offline)", "by_score": tiers}
        del layers, ws, x, bufs
        torch.cuda.empty_cache()

    if want("predictor"):
        # ---- low-rank gate predictor on the Llama shape (sffn_decode_predicted):
        # random rank-256 fp32 factors (timing only: quality needs trained weights),
        # A scaled so that A (B x) spreads like the gate bias; alpha per layer so a
        # target share of the timed tokens' neurons are candidates
        c = W.CONFIGS[2]
        F, d, nl, rank = c["d_ff"], c["d_model"], c["layers"], 256
        layers, ws, x, bufs = setup(2, nl, norms=False)
        gen = torch.Generator(device=dev).manual_seed(11)
        xt = x[:T].float()
        facs, preds = [], []
        for l in range(nl):
            A = torch.randn(F, rank, generator=gen, device=dev) / rank ** 0.5
            Bf = torch.randn(rank, d, generator=gen, device=dev) / d ** 0.5
            q = (xt @ Bf.t()) @ A.t()
            A = (A * (0.5 / q.std())).contiguous()
            bias = layers[l]["b_gate"].to(dev).float()
            facs.append((A, Bf.contiguous()))
            preds.append((xt @ Bf.t()) @ A.t() + bias[None, :])
        exact_us = run_sparse(ws, x, bufs, 1, sffn.MODE_EXACT, sffn.SCORE_GATE, [0.0] * nl)
        lr = {"workload": "llama2-7b-reglu shape (d_model 4096, d_ff 11008 bf16, 8 layers), B=1, rank-256 fp32 "
                          "factors (random: timing only), exact rule on the candidates",
              "exact_decode_us_per_token": round(exact_us, 3), "points": []}
        for frac in (0.15, 0.3, 0.5):
            alphas, cand = [], []
            for l in range(nl):
                v = torch.quantile(preds[l][l::nl].flatten(), 1.0 - frac).item()
                alphas.append(max(0.0, -v))
                cand.append((preds[l][l::nl] >= -alphas[-1]).float().mean().item())

            def enq():
                for t in range(T):
                    A, Bf = facs[t % nl]
                    sffn.decode_predicted(x[t:t + 1], ws[t % nl], A, Bf, alphas[t % nl], out=bufs["o"][t:t + 1],
                                          active_idx=bufs["idx"][t:t + 1], n_active=bufs["n"][t:t + 1],
                                          workspace=bufs["work"], stream=stream)
            us = _time_graph(enq, stream, max(3, args.steps // 3), args.warmup) * 1e3 / T
            a = float(bufs["n"][:T].float().mean().item()) / F
            cf = sum(cand) / nl
            nbytes = 4.0 * rank * (F + d) + rowb(c) * F * (cf + 2 * a)
            lr["points"].append(point(us, nbytes, candidates=round(cf, 4), a=round(a, 4),
                                      speedup_vs_exact=round(exact_us / us, 3)))
        out["lowrank_predictor"] = lr
        del layers, ws, x, bufs, facs, preds
        torch.cuda.empty_cache()

    if want("tiny"):
        # ---- tiny fp32 ReGLU layer (L2 resident, launch bound: us/token only)
        layers, ws, x, bufs = setup(1, 1, norms=False)
        us = run_sparse(ws, x, bufs, 1, sffn.MODE_EXACT, sffn.SCORE_GATE, [0.0])
        out["tiny_fp32"] = {"us_per_token": round(us, 3), "a": round(float(bufs["n"].float().mean().item()) / 688, 4)}
    return out


def traffic_for(key):
    """DRAM bytes per launch from a committed ncu capture, or None if the kernel
    sources changed since it was taken (profiles/traffic.json holds the hash)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(key)
        if not e:
            return None
        h = hashlib.sha256()
        for f in e["sources"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        return e["bytes"] if h.hexdigest() == e["sha256"] else None
    except Exception:
        return None


def bench_moe(args, dev):
    """MoE routing and block budget on the prefill workload's sequence: the
    adaptive top-K of 16384 tokens over 384 routed experts (a layer of the
    16-39 range: cap 5), and the 128-token block budget of the L 16384,
    d_model 5120 sequence at mass 0.5."""
    import torch

    from activation_sparse_ffn_gemv_gb300 import sffn
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    hbm, _, _, _ = peaks()
    T, E = 16384, 384
    g = torch.Generator(device=dev).manual_seed(3)
    logits = [torch.randn(T, E, generator=g, device=dev) * 1.5 for _ in range(4)]  # 4 x 25 MB: beyond L2
    cap = sffn.moe_progressive_k(20)
    k = torch.empty(T, dtype=torch.int32, device=dev)
    ex = torch.empty((T, cap), dtype=torch.int32, device=dev)
    wt = torch.empty((T, cap), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def enq():
        for i in range(4):
            sffn.moe_route(logits[i], cap, 0.5, k_out=k, experts=ex, weights=wt, stream=stream)
    ms = _time_graph(enq, stream, max(5, args.steps), args.warmup) / 4
    nbytes = T * E * 4 + T * (4 + 8 * cap)
    gbps = nbytes / (ms * 1e-3) / 1e9
    route = {"workload": f"{T} tokens x {E} routed experts fp32 logits, layer 20 (cap {cap}), buckets (3,4,5,6), "
                         "mass 0.5", "ms": round(ms, 4), "gbps": round(gbps, 1), "frac_hbm": round(gbps / hbm, 4),
             "mean_k": round(float(k.float().mean().item()), 3)}
    c = W.CONFIGS[5]
    L, d = c["L"], c["d_model"]
    _, Ya = W.make_prefill_inputs(L, d, seed=0, device=dev)
    nb = (L + 127) // 128
    ti = torch.empty(L, dtype=torch.int32, device=dev)
    nt = torch.empty(1, dtype=torch.int32, device=dev)
    rg = torch.empty((nb, 2), dtype=torch.int32, device=dev)
    nr = torch.empty(1, dtype=torch.int32, device=dev)
    wsb = torch.empty(sffn.lib().sffn_moe_budget_workspace_size(L, d), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def enq2():
        sffn.moe_block_budget(Ya, 0.5, token_idx=ti, n_tokens=nt, ranges=rg, n_ranges=nr, workspace=wsb,
                              stream=stream)
    ms2 = _time_graph(enq2, stream, max(5, args.steps), args.warmup)
    budget = {"workload": f"L {L}, d_model {d} bf16 attention outputs, mass 0.5, ratios [0.10, 0.50], 128-token "
                          "blocks", "ms": round(ms2, 4), "tokens": int(nt.item()), "ranges": int(nr.item())}
    return {"route": route, "block_budget": budget}


def bench_prefill_stack(args, dev):
    """Four prefill layers of the token-selective configuration through the
    per-layer schedule (layer 0 dense, layers 1-2 mass 0.5, layer 3 mass 0.2)
    against the same four layers all dense, one CUDA graph per stack."""
    import torch

    from activation_sparse_ffn_gemv_gb300 import sffn
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    try:
        c = W.CONFIGS[5]
        L, d, n = c["L"], c["d_model"], 4
        layers = [W.make_ffn_layer(5, seed=300 + i, layer=i, device=dev) for i in range(n)]
        ws = [sffn.Weights(layer) for layer in layers]
        X, _ = W.make_prefill_inputs(L, d, seed=3, device=dev)
        yas = [W.make_prefill_inputs(L, d, seed=40 + i, device=dev)[1] for i in range(n)]
        stream = torch.cuda.Stream(device=dev)
        nb = max(int(sffn.lib().sffn_prefill_layers_workspace_size(L, w.ref())) for w in ws)
        wsp = torch.zeros(nb, dtype=torch.uint8, device=dev)
        out = torch.empty_like(X)
        sel = torch.empty((n, L), dtype=torch.int32, device=dev)
        ns = torch.empty(n, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()  # made on the default stream, used on `stream`
        res = {"workload": "4 token-selective prefill layers (L 16384, d_model 5120, d_ff 25600, SwiGLU bf16); "
                           "schedule: layer 0 dense, layers 1-2 mass 0.5, layer 3 mass 0.2, recent_n 128, "
                           "min_keep 1; synthetic attention outputs per layer"}
        scheds = (("scheduled", sffn.schedule(dense_until=1, mass_thresh=0.5, recent_n=c["recent_n"],
                                              min_keep=c["min_keep"], deep_layer_start=3, mass_thresh_deep=0.2)),
                  ("dense", sffn.schedule_preset("dense")))
        for name, sch in scheds:
            def enq(sch=sch):
                sffn.prefill_layers(X, yas, ws, sch, out=out, sel_idx=sel, n_sel=ns, workspace=wsp, stream=stream)
            ms = _time_graph(enq, stream, max(2, args.prefill_steps // 2), args.warmup)
            res[name] = {"ms_per_stack": round(ms, 4), "tokens_per_s": round(L / (ms * 1e-3)),
                         "n_sel_per_layer": ns.tolist()}
        res["speedup_vs_dense"] = round(res["dense"]["ms_per_stack"] / res["scheduled"]["ms_per_stack"], 3)
        del layers, ws, yas
        torch.cuda.empty_cache()
        return res
    except Exception as e:  # reported in the JSON line; the other measurements stand
        torch.cuda.empty_cache()
        return {"error": f"{type(e).__name__}: {e}"}


def bench_prefill(args, dev, rank, world, dist):
    """Token-selective prefill (L 16384, d_model 5120, d_ff 25600, SwiGLU bf16):
    token selection + the selected-token FFN, at each mass threshold."""
    import torch

    from activation_sparse_ffn_gemv_gb300 import sffn
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    c = W.CONFIGS[5]
    L, d, F = c["L"], c["d_model"], c["d_ff"]
    layer = W.make_ffn_layer(5, seed=7 + rank, device=dev)
    X, Ya = W.make_prefill_inputs(L, d, seed=rank, device=dev)
    w = sffn.Weights(layer)
    ws_sel = sffn.alloc_workspace(sffn.WS_SELECT, L, None, dev)
    ws_pf = sffn.alloc_workspace(sffn.WS_PREFILL, L, w, dev)
    sel = torch.empty(L, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(X)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()  # made on the default stream, used on `stream`
    _, bf16_peak, _, peak_src = peaks()
    rows = {}
    for m in c["mass"]:
        def sel_call():
            sffn.token_select(Ya, m, c["recent_n"], c["min_keep"], sel_idx=sel, n_sel=n, workspace=ws_sel,
                              stream=stream)

        def ffn_call():
            sffn.prefill(X, Ya, w, sel, n, out=out, workspace=ws_pf, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                sel_call()
                ffn_call()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.prefill_steps + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(args.prefill_steps):
                sel_call()
                ev[2 * i + 1].record(stream)
                ffn_call()
                ev[2 * i + 2].record(stream)
        ev[-1].synchronize()
        t_sel = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.prefill_steps)) / args.prefill_steps
        t_ffn = sum(ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(args.prefill_steps)) / args.prefill_steps
        t_tot = ev[0].elapsed_time(ev[-1]) / args.prefill_steps
        t_tot, t_ffn, t_sel = max_over_ranks([t_tot, t_ffn, t_sel], dist, dev)
        k = int(n.item())
        flops = 6.0 * k * d * F
        tf = flops / (t_ffn * 1e-3) / 1e12
        rows[str(m)] = {"n_sel": k, "select_ms": round(t_sel, 4), "ffn_ms": round(t_ffn, 4),
                        "tokens_per_s": round(world * L / (t_tot * 1e-3)),
                        "ffn_tflops": round(tf, 1), "ffn_frac_bf16_peak": round(tf / bf16_peak, 4)}
    res = {"metric": "sparse-prefill tokens/s", "unit": "tokens/s",
           "workload": "token-selective-prefill: L 16384, d_model 5120, d_ff 25600, SwiGLU bf16, recent_n 128, "
                       "min_keep 1, Y_attn rows scaled by exp(N(0,1))",
           "value": rows["0.2"]["tokens_per_s"], "by_mass": rows,
           "speedup_vs_dense": round(rows["0.2"]["tokens_per_s"] / rows["1.0"]["tokens_per_s"], 3),
           "roofline": {"bound": "tensor", "kernel": "sffn_prefill FFN (tcgen05 SwiGLU + down GEMMs), mass 0.5",
                        "achieved": rows["0.5"]["ffn_tflops"], "peak": bf16_peak, "unit": "TFLOP/s",
                        "frac": rows["0.5"]["ffn_frac_bf16_peak"], "peak_source": peak_src,
                        "flops_per_launch": 6.0 * rows["0.5"]["n_sel"] * d * F,
                        "traffic": traffic_for("prefill_m05")}}
    # the same selection with int4-g64 weights (the write-up's INT4 setting)
    layer4 = W.make_ffn_layer(4, seed=7 + rank, d_model=d, d_ff=F, device=dev)
    w4 = sffn.Weights(layer4)
    ws4 = sffn.alloc_workspace(sffn.WS_PREFILL, L, w4, dev)
    torch.cuda.synchronize()
    rows4 = {}
    for m in (0.2, 0.5, 1.0):
        sffn.token_select(Ya, m, c["recent_n"], c["min_keep"], sel_idx=sel, n_sel=n, workspace=ws_sel, stream=stream)

        def ffn4():
            sffn.prefill(X, Ya, w4, sel, n, out=out, workspace=ws4, stream=stream)
        ms = _time_graph(ffn4, stream, args.prefill_steps, args.warmup)
        k = int(n.item())
        tf = 6.0 * k * d * F / (ms * 1e-3) / 1e12
        rows4[str(m)] = {"n_sel": k, "ffn_ms": round(ms, 4), "ffn_tflops": round(tf, 1),
                         "ffn_frac_bf16_peak": round(tf / bf16_peak, 4),
                         "ffn_vs_bf16": round(rows[str(m)]["ffn_ms"] / ms, 3)}
    res["int4_g64"] = {"workload": "the same layer shape with int4-g64 weights (codes U{-8..7}, fp16 group "
                                   "scales), dequantised to bf16 tiles inside the GEMMs", "by_mass": rows4}
    del layer4, w4, ws4
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(layer, X, Ya)
    return res


def prefill_cpu_baseline(layer_dev, X, Ya, nrows=8):
    import numpy as np

    import oracle as O
    from tests.oracle_io import ffn_from_layer, mat_from_act
    layer = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in layer_dev.items()}
    Xc, Yc = X.cpu(), Ya.cpu()
    L = Xc.shape[0]
    mask = np.ones(L, np.uint8)
    rows = np.arange(0, L, L // nrows, dtype=np.int32)[:nrows]
    nth = min(os.cpu_count() or 1, nrows)
    t0 = time.perf_counter()
    O.prefill_rows(ffn_from_layer(layer), mat_from_act(Xc), mat_from_act(Yc), mask, rows, nthreads=nth)
    dt = time.perf_counter() - t0
    return {"value": round(nrows / dt, 3), "unit": "selected rows/s", "cores": nth, "kind": "oracle",
            "sample": f"{nrows} selected rows of the prefill FFN, fp64 oracle, {nth} threads"}


def cpu_baseline(layer_dev, x_cpu, nthreads=None):
    import oracle as O
    from tests.oracle_io import ffn_from_layer, mat_from_act
    layer = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in layer_dev.items()}
    nthreads = nthreads or os.cpu_count() or 1
    ffn, xm = ffn_from_layer(layer), mat_from_act(x_cpu)
    t0 = time.perf_counter()
    O.decode(ffn, xm, O.EXACT, nthreads=nthreads)
    dt = time.perf_counter() - t0
    n = x_cpu.shape[0]
    return {"value": round(dt * 1e6 / n, 1), "unit": "us/token", "cores": int(nthreads), "kind": "oracle",
            "sample": f"{n} tokens of the same workload (layer copy 0), exact gating, fp64 oracle, "
                      f"{nthreads} threads over tokens"}


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return None
    import torch

    import oracle as O
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    from tests.oracle_io import ffn_from_layer, mat_from_act
    O.build()
    cfg = W.CONFIGS[2]
    layer = W.make_ffn_layer(2, seed=0, layer=0)
    nthreads = os.cpu_count() or 1
    per_step = max(1, min(nthreads, 16))
    x = W.make_tokens(2, per_step * (args.warmup + args.steps), seed=0)
    ffn = ffn_from_layer(layer)
    for i in range(args.warmup):
        O.decode(ffn, mat_from_act(x[i * per_step:(i + 1) * per_step]), O.EXACT, nthreads=nthreads)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        O.decode(ffn, mat_from_act(x[i * per_step:(i + 1) * per_step]), O.EXACT, nthreads=nthreads)
    dt = time.perf_counter() - t0
    us_tok = dt * 1e6 / (args.steps * per_step)
    return {
        "impl": "reference", "metric": METRIC, "value": round(us_tok, 1), "unit": "us/token", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1/d_in) weights, gate bias N(-1.2,0.3), x N(0,1)",
        "config": {"workload": "llama2-7b-reglu-decode: d_model 4096, d_ff 11008, bf16, exact gating, "
                               "batch 1, bounded sample per step",
                   "d_model": cfg["d_model"], "d_ff": cfg["d_ff"], "batch": 1, "tokens_per_step": per_step},
        "cpu_baseline": {"value": round(us_tok, 1), "unit": "us/token", "cores": nthreads, "kind": "oracle",
                         "sample": f"{per_step} tokens per step, layer copy 0, fp64 oracle"},
        "e2e": {"value": round(us_tok, 1), "unit": "us/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=1024)
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-sweeps", action="store_true")
    ap.add_argument("--sweep", default=None,
                    help="comma-separated decode workload legs to run (int4, batch, keep_ratio, predictor, tiny); "
                         "default all")
    ap.add_argument("--no-decode", action="store_true", help="run only the prefill leg (profiling)")
    ap.add_argument("--prefill-steps", type=int, default=10)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        res = run_reference(args)
    elif args.no_decode:
        res = run_prefill_only(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
