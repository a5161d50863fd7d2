"""Benchmark of the DiT block's projection hot path on GB300.

One step = the four dynamic-LoRA NVFP4 projections of one transformer block
at packed sequence length S = 37726 (fused QKV 5120->15360 rank 384,
attention-out 5120->5120, fused gate/up 5120->27648 with SiLU*up, down
13824->5120, ranks 128, alpha = rank, strength 1), run back to back on one
stream through the C ABI; down consumes gate/up's output.  Inputs are seeded
synthetic tensors already resident in HBM (each activation is larger than L2,
so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded row x column sample of the same workload on the host cores.
"""
from __future__ import annotations

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

from nvfp4_linear_lora_gb300 import configs, synth  # noqa: E402


# DRAM traffic of the GEMM launches (dram__bytes_read.sum + dram__bytes_write.sum
# per launch) of the block, from one ncu capture at S=16384 (the timed step's
# four launches; a capture at full size would exceed the size rule for a
# multi-pass capture) scaled by the rows, 37726 / 16384: every term of a
# launch's traffic (x panels, output, the weight once per raster group) grows
# with M.  Summarised in profiles/dram_fp4gemm_pair_S16384.md.  It is reported
# only while the GEMM sources hash to the value the capture was taken with;
# after any change to them the counters no longer describe the kernel and
# `traffic` is null.
GEMM_TRAFFIC = {"sources_sha256": "0a254c438c5c3a314eef515553d32f6e101c71e812e6331230b39a502417cbd7", "S": 37726,
                "scaled_from": {"S": 16384, "bytes_per_launch": {"qkv": 217108480 + 468796160,
                                                                 "attn_out": 67608576 + 119828480,
                                                                 "gate_up": 232174592 + 419132928,
                                                                 "down": 252185600 + 148391680}},
                "bytes_per_launch": {k: round(v * 37726 / 16384) for k, v in
                                     {"qkv": 217108480 + 468796160, "attn_out": 67608576 + 119828480,
                                      "gate_up": 232174592 + 419132928, "down": 252185600 + 148391680}.items()}}
GEMM_SOURCES = ("nvfp4_linear_lora_gb300/csrc/h3lin_gemm.cu", "nvfp4_linear_lora_gb300/csrc/h3lin_device.cuh")


def gemm_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    here = os.path.dirname(os.path.abspath(__file__))
    for rel in GEMM_SOURCES:
        with open(os.path.join(here, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_algorithmic_bytes(S):
    """Bytes one GEMM launch must move at least: x codes + scales, W codes +
    scales, u and B' (bf16), the bf16 output."""
    out = {}
    for name, K, N, r, silu in configs.BLOCK_PROJECTIONS:
        n_out = N // 2 if silu else N
        out[name] = S * K // 2 + S * K // 16 + N * K // 2 + N * K // 16 + 2 * S * r + 2 * N * r + 2 * S * n_out
    return out

METRIC = "NVFP4+LoRA projection TFLOP/s at S=37726 (% of dense FP4 peak); ms/block"
FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense FP4 : BF16 tensor ratio on GB300
FP4_NOMINAL_TFLOPS = 13500.0      # GB300 datasheet dense FP4 (no sparsity), for context next to the measured-derived peak
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--S", type=int, default=configs.BLOCK_S)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-merged", action="store_true",
                    help="skip the merged-LoRA comparison (weights with the adapter folded in, base path only)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU-oracle sample time")
    ap.add_argument("--no-modulation", action="store_true",
                    help="skip the modulation-producer measurement on the block's QKV input")
    ap.add_argument("--no-rope", action="store_true",
                    help="skip the Q/K RMSNorm + RoPE measurement on the block's QKV output")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sequence-length sweep of the QKV projection (M = 1024 ... 65536)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-projection workloads (tiny, QKV M=9437, adapter switching at S=37728)")
    ap.add_argument("--unfused-mlp", action="store_true",
                    help="run gate/up and down as two plain projections (amax pass over h) instead of the "
                         "MLP's producer fusion")
    return ap.parse_args(argv)


def max_over_ranks(ms, world, device):
    """The slowest rank's time: every rank contributes its own, all get the max
    (replicas: the job is done when the last one is)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, ms):
    """Whole-job throughput: every rank processes its own block (weak scaling)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def block_flops(S):
    """(total, base FP4, LoRA down, LoRA up) algorithmic FLOPs of one block."""
    base = down = up = 0
    for _, K, N, r, _ in configs.BLOCK_PROJECTIONS:
        base += 2 * S * K * N
        down += 2 * S * K * r
        up += 2 * S * r * N
    return base + down + up, base, down, up


# ----------------------------------------------------------------- workload
def make_block_inputs(S, seed=configs.BLOCK_SEED):
    """Host inputs of the block, one generator in block order: per projection
    x (not for down, which consumes gate/up's output), s, W, A, B."""
    rng = np.random.default_rng(seed)
    out = []
    for name, K, N, r, silu in configs.BLOCK_PROJECTIONS:
        x = synth.activation(rng, S, K) if name != "down" else None
        s = synth.pre_quant_scale(rng, K)
        W = synth.weight(rng, N, K)
        ad = synth.adapter(rng, N, K, r)
        out.append(dict(name=name, K=K, N=N, rank=r, silu=silu, x=x, pqs=s, W=W, adapter=ad))
    return out


class Block:
    """Device-resident block: packed weights, adapters, workspaces, outputs.

    With ``fused_mlp`` (the default) gate/up and down run as the MLP's
    producer fusion: gate/up's epilogue leaves amax(h * s_down) in down's
    workspace and down's prepare is one pass over h (h3lin_mlp_forward, or its
    stages when the GEMMs are timed); the results are bit-identical to the
    unfused chain."""

    def __init__(self, host, S, device, fused_mlp=True):
        import torch

        from nvfp4_linear_lora_gb300 import h3lin
        self.h3lin = h3lin
        self.S = S
        self.proj = []
        stream = torch.cuda.current_stream().cuda_stream
        for p in host:
            d = dict(p)
            d["x_dev"] = synth.to_bf16_tensor(p["x"]).to(device) if p["x"] is not None else None
            d["pqs_dev"] = torch.from_numpy(p["pqs"]).to(device)
            Wd = synth.to_bf16_tensor(p["W"]).to(device)
            d["pw"] = h3lin.pack_weight(Wd)
            del Wd
            a = p["adapter"]
            d["ad"] = h3lin.Adapter(synth.to_bf16_tensor(a["A"]).to(device), synth.to_bf16_tensor(a["B"]).to(device),
                                    a["rank"], a["alpha"])
            n_out = p["N"] // 2 if p["silu"] else p["N"]
            d["out"] = torch.empty((S, n_out), dtype=torch.bfloat16, device=device)
            wsb = h3lin.h3lin_forward_workspace_bytes(S, p["K"], p["N"], p["rank"])
            d["ws"] = h3lin.new_workspace(wsb, device)
            d["wc"] = d["pw"].c_struct()
            d["ac"] = d["ad"].c_struct()
            d["stream"] = stream
            self.proj.append(d)
        # down consumes gate/up's output
        self.proj[3]["x_dev"] = self.proj[2]["out"]
        self.fused_mlp = fused_mlp
        if fused_mlp:   # down's workspace also serves h3lin_mlp_forward (both projections)
            gu, dn = self.proj[2], self.proj[3]
            wsb = h3lin.h3lin_mlp_workspace_bytes(S, gu["K"], gu["N"], dn["N"], max(gu["rank"], dn["rank"]))
            dn["ws"] = h3lin.new_workspace(wsb, device)
        torch.cuda.synchronize()

    def launches_per_step(self):
        # per projection: amax (+ A(x)), quantise, GEMM; the fused MLP's down
        # projection has one pass (quantise + A(h)) instead of two
        return 3 * len(self.proj) - (1 if self.fused_mlp else 0)

    def _mlp(self):
        h, gu, dn = self.h3lin, self.proj[2], self.proj[3]
        st = h.h3lin_mlp_forward(gu["x_dev"].data_ptr(), self.S, gu["pqs_dev"].data_ptr(), gu["wc"], gu["ac"], 1.0,
                                 dn["pqs_dev"].data_ptr(), dn["wc"], dn["ac"], 1.0, gu["out"].data_ptr(),
                                 dn["out"].data_ptr(), h.H3LIN_OUT_BF16, dn["ws"].data_ptr(), dn["ws"].numel(),
                                 dn["stream"])
        if st:
            raise h.H3linError(st, "h3lin_mlp_forward")

    def step(self, gemm_events=None):
        """One block.  With ``gemm_events`` (list of (start, stop) per
        projection) the two stages are enqueued separately with events around
        the GEMM kernel, on the same stream."""
        h = self.h3lin
        for i, d in enumerate(self.proj):
            fuse = self.fused_mlp and i >= 2
            if fuse and gemm_events is None:
                if i == 2:
                    self._mlp()
                continue
            if gemm_events is None:
                st = h.h3lin_forward(d["x_dev"].data_ptr(), self.S, d["pqs_dev"].data_ptr(), d["wc"],
                                     h.H3LIN_EPI_SILU_MUL if d["silu"] else h.H3LIN_EPI_NONE, d["ac"], 1.0,
                                     d["out"].data_ptr(), h.H3LIN_OUT_BF16, d["ws"].data_ptr(), d["ws"].numel(),
                                     d["stream"])
                if st:
                    raise h.H3linError(st, "h3lin_forward")
            else:
                prep = h.h3lin_forward_prepare_produced if (fuse and i == 3) else h.h3lin_forward_prepare
                st = prep(d["x_dev"].data_ptr(), self.S, d["pqs_dev"].data_ptr(), d["wc"], d["ac"], 1.0,
                          d["ws"].data_ptr(), d["ws"].numel(), d["stream"])
                if st:
                    raise h.H3linError(st, "h3lin_forward_prepare")
                gemm_events[i][0].record()
                epi = h.H3LIN_EPI_SILU_MUL if d["silu"] else h.H3LIN_EPI_NONE
                if fuse and i == 2:   # producer: amax of h for down, into down's workspace
                    nx = self.proj[3]
                    st = h.h3lin_forward_gemm_produce(self.S, d["wc"], epi, d["ac"], 1.0, d["out"].data_ptr(),
                                                      d["ws"].data_ptr(), d["ws"].numel(),
                                                      nx["pqs_dev"].data_ptr(), nx["ws"].data_ptr(),
                                                      nx["ws"].numel(), d["stream"])
                else:
                    st = h.h3lin_forward_gemm(self.S, d["wc"], epi, d["ac"], 1.0, d["out"].data_ptr(),
                                              h.H3LIN_OUT_BF16, d["ws"].data_ptr(), d["ws"].numel(), d["stream"])
                if st:
                    raise h.H3linError(st, "h3lin_forward_gemm")
                gemm_events[i][1].record()

    def step_io(self, xs, outs):
        """One block reading x1, x2, x3 from ``xs`` and writing the QKV,
        attn-out and down outputs into ``outs`` (gate/up's h stays internal)."""
        saved = [(d["x_dev"], d["out"]) for d in self.proj]
        try:
            for d, x in zip(self.proj[:3], xs):
                d["x_dev"] = x
            for d, o in zip((self.proj[0], self.proj[1], self.proj[3]), outs):
                d["out"] = o
            self.step()
        finally:
            for d, (x, o) in zip(self.proj, saved):
                d["x_dev"], d["out"] = x, o

    def check_status(self):
        for d in self.proj:
            v = self.h3lin.read_status(d["ws"])
            if v != 0:
                raise RuntimeError(f"device status {v} in projection {d['name']}")



# ------------------------------------------------------- single projections
def gemm_roofline(base_flops, lup_flops, gemm_ms, peaks):
    """The GEMM's mixed FP4/BF16 roofline: ideal time at the burst peaks
    (measured bf16 x the nominal FP4:BF16 ratio for the FP4 part)."""
    peak_bf16 = peaks["bf16_tflops"]
    peak_fp4 = peak_bf16 * FP4_OVER_BF16
    ideal_s = base_flops / (peak_fp4 * 1e12) + lup_flops / (peak_bf16 * 1e12)
    mixed = (base_flops + lup_flops) / ideal_s / 1e12
    achieved = (base_flops + lup_flops) / (gemm_ms * 1e-3) / 1e12
    return {"achieved": achieved, "peak": mixed, "unit": "TFLOP/s", "frac": achieved / mixed}


class Projection:
    """One projection resident on the device: x, pre_quant_scale, packed
    weight, resident adapters, output and workspace."""

    def __init__(self, x, pqs, W, adapters, silu, device, max_rank=None):
        import torch

        from nvfp4_linear_lora_gb300 import h3lin
        self.h3lin = h3lin
        self.M, self.K = x.shape
        self.N = W.shape[0]
        self.silu = silu
        self.x = synth.to_bf16_tensor(x).to(device)
        self.pqs = torch.from_numpy(pqs).to(device)
        Wd = synth.to_bf16_tensor(W).to(device)
        self.pw = h3lin.pack_weight(Wd)
        del Wd
        self.ads = [h3lin.Adapter(synth.to_bf16_tensor(a["A"]).to(device), synth.to_bf16_tensor(a["B"]).to(device),
                                  a["rank"], a["alpha"]) for a in adapters]
        self.acs = [a.c_struct() for a in self.ads]
        self.wc = self.pw.c_struct()
        r = max_rank if max_rank is not None else max([a["rank"] for a in adapters] + [0])
        self.out = torch.empty((self.M, self.N // 2 if silu else self.N), dtype=torch.bfloat16, device=device)
        self.ws = h3lin.new_workspace(h3lin.h3lin_forward_workspace_bytes(self.M, self.K, self.N, r), device)
        self.stream = torch.cuda.current_stream().cuda_stream

    def flops(self, adapter_index, strength):
        f = 2 * self.M * self.K * self.N
        if adapter_index is not None and strength != 0.0:
            r = self.ads[adapter_index].rank
            f += 2 * self.M * self.K * r + 2 * self.M * r * self.N
        return f

    def lora_up_flops(self, adapter_index, strength):
        if adapter_index is None or strength == 0.0:
            return 0
        return 2 * self.M * self.ads[adapter_index].rank * self.N

    def run(self, adapter_index=0, strength=1.0, gemm_event=None):
        h = self.h3lin
        ac = self.acs[adapter_index] if adapter_index is not None else None
        epi = h.H3LIN_EPI_SILU_MUL if self.silu else h.H3LIN_EPI_NONE
        if gemm_event is None:
            st = h.h3lin_forward(self.x.data_ptr(), self.M, self.pqs.data_ptr(), self.wc, epi, ac, strength,
                                 self.out.data_ptr(), h.H3LIN_OUT_BF16, self.ws.data_ptr(), self.ws.numel(),
                                 self.stream)
            if st:
                raise h.H3linError(st, "h3lin_forward")
            return
        st = h.h3lin_forward_prepare(self.x.data_ptr(), self.M, self.pqs.data_ptr(), self.wc, ac, strength,
                                     self.ws.data_ptr(), self.ws.numel(), self.stream)
        if st:
            raise h.H3linError(st, "h3lin_forward_prepare")
        gemm_event[0].record()
        st = h.h3lin_forward_gemm(self.M, self.wc, epi, ac, strength, self.out.data_ptr(), h.H3LIN_OUT_BF16,
                                  self.ws.data_ptr(), self.ws.numel(), self.stream)
        if st:
            raise h.H3linError(st, "h3lin_forward_gemm")
        gemm_event[1].record()

    def check_status(self):
        v = self.h3lin.read_status(self.ws)
        if v != 0:
            raise RuntimeError(f"device status {v}")


def time_calls(proj, calls, steps, warmup):
    """Run the call list (adapter index or None, strength) `steps` times after
    `warmup` untimed rounds; CUDA events around the whole region and around
    every GEMM.  Returns (ms per round, GEMM ms per round)."""
    import torch
    for _ in range(warmup):
        for ai, sv in calls:
            proj.run(ai, sv)
    torch.cuda.synchronize()
    proj.check_status()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for k in range(steps):
        for j, (ai, sv) in enumerate(calls):
            proj.run(ai, sv, ev[k][j])
    t1.record()
    torch.cuda.synchronize()
    proj.check_status()
    gemm = sum(statistics.mean(ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(steps))
               for j in range(len(calls)))
    return t0.elapsed_time(t1) / steps, gemm


def oracle_projection_sample(x, pqs, W, adapter, silu, m_rows, n_cols, seed):
    """The oracle on a row x output-column sample of one projection: (seconds, flops)."""
    from oracle import linear
    rng = np.random.default_rng(seed)
    N, K = W.shape
    if silu:
        c = np.sort(rng.choice(N // 2, min(n_cols // 2, N // 2), replace=False))
        cols = np.concatenate([c, c + N // 2])
    else:
        cols = np.sort(rng.choice(N, min(n_cols, N), replace=False))
    rows = np.sort(rng.choice(x.shape[0], min(m_rows, x.shape[0]), replace=False))
    t0 = time.perf_counter()
    wq, ws, tsw = linear.pack_weight(W[cols])
    ad = None
    if adapter is not None:
        ad = dict(adapter)
        ad["B"] = adapter["B"][cols]
    linear.forward(x[rows], (wq, ws, tsw), pqs, ad, 1.0, silu)
    dt = time.perf_counter() - t0
    r = adapter["rank"] if adapter is not None else 0
    return dt, 2 * len(rows) * (K * len(cols) + K * r + r * len(cols))


def projection_line(name, proj, calls, steps, warmup, peaks, host=None, what=""):
    """One workload's JSON object: ms, TFLOP/s, the GEMM's roofline, and
    (with host inputs) the oracle on a small sample of the same workload."""
    ms, gemm_ms = time_calls(proj, calls, steps, warmup)
    flops = sum(proj.flops(ai, sv) for ai, sv in calls)
    base = 2 * proj.M * proj.K * proj.N * len(calls)
    lup = sum(proj.lora_up_flops(ai, sv) for ai, sv in calls)
    line = {"workload": name, "M": proj.M, "K": proj.K, "N": proj.N, "calls_per_step": len(calls),
            "ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "frac_of_fp4_peak": flops / (ms * 1e-3) / 1e12 / (peaks["bf16_tflops"] * FP4_OVER_BF16),
            "gemm_ms_per_step": gemm_ms, "prepare_ms_per_step": ms - gemm_ms,
            "roofline": dict(kernel="k_fp4gemm", bound="tensor", **gemm_roofline(base, lup, gemm_ms, peaks)),
            "what": what}
    if host is not None:
        x, pqs, W, adapter, silu = host
        t, f = oracle_projection_sample(x, pqs, W, adapter, silu, 64, 512, seed=proj.M)
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cpu_info(), "kind": "oracle",
                                "sample": f"64 rows x 512 output columns, {t:.2f} s"}
    return line


def _tiny_inputs():
    t = configs.TINY
    p = synth.projection(t["seed"], t["M"], t["K"], t["N"], t["rank"])
    return p["x"], p["pqs"], p["W"], [p["adapter"]]


def _qkv_inputs():
    q = configs.QKV
    p = synth.projection(q["seed"], q["M"], q["K"], q["N"], q["rank"], outlier_frac=q["outlier_frac"])
    return p["x"], p["pqs"], p["W"], [p["adapter"]]


def _switch_inputs():
    # two resident adapters (rank 384 and 128, their own seeds) on the QKV shape at S = 37728
    rng = np.random.default_rng(configs.SWITCH_SEED)
    K, N = configs.HIDDEN, 3 * configs.HIDDEN
    x = synth.activation(rng, configs.SWITCH_S, K, "normal", 0.01)
    s = synth.pre_quant_scale(rng, K)
    W = synth.weight(rng, N, K)
    ads = [synth.adapter(np.random.default_rng(sd), N, K, r) for sd, r in zip(configs.SWITCH_ADAPTER_SEEDS, (384, 128))]
    return x, s, W, ads


def _sweep_inputs(M, seed):
    K, N, r = configs.HIDDEN, 3 * configs.HIDDEN, 384
    rng = np.random.default_rng(seed)
    x = synth.activation(rng, M, K, "student_t3", 0.01)
    s = synth.pre_quant_scale(rng, K)
    W = synth.weight(rng, N, K)
    return x, s, W, [synth.adapter(rng, N, K, r)]


def start_workload_inputs(a, pool):
    """Host inputs of the single-projection workloads, drawn on worker threads
    (each from its own seeded generator) while the block is set up and timed."""
    futs = {}
    if not a.no_configs:
        futs["tiny"] = pool.submit(_tiny_inputs)
        futs["qkv_9437"] = pool.submit(_qkv_inputs)
        futs["switch_S37728"] = pool.submit(_switch_inputs)
    if not a.no_sweep:
        for M, seed in zip(configs.SWEEP_M, configs.SWEEP_SEEDS):
            futs[f"sweep_M{M}"] = pool.submit(_sweep_inputs, M, seed)
    return futs


def workload_lines(a, device, peaks, futs):
    """Throughput on the single-projection workloads (the tiny projection, the
    QKV projection at M = 9437, adapter switching at S = 37728) and the
    sequence-length sweep of the QKV projection."""
    import torch
    steps, warmup = max(5, a.steps // 10), 3
    out = {}
    if not a.no_configs:
        x, s, W, ads = futs.pop("tiny").result()
        pr = Projection(x, s, W, ads, False, device)
        out["tiny"] = projection_line("tiny", pr, [(0, 1.0)], steps, warmup, peaks, host=(x, s, W, ads[0], False),
                                      what="M=200 K=256 N=384 rank 16 (launch-bound: three kernels for 0.04 GFLOP)")
        x, s, W, ads = futs.pop("qkv_9437").result()
        pr = Projection(x, s, W, ads, False, device)
        out["qkv_9437"] = projection_line("qkv_9437", pr, [(0, 1.0)], steps, warmup, peaks,
                                          host=(x, s, W, ads[0], False),
                                          what="fused QKV 5120->15360 rank 384, M=9437 (ragged), 1% outlier channels")
        del pr
        x, s, W, ads = futs.pop("switch_S37728").result()
        pr = Projection(x, s, W, ads, False, device)
        calls = [(0, 1.0), (1, 0.5), (None, 1.0), (0, 0.0), (1, 1.0), (0, 0.5)]
        out["switch_S37728"] = projection_line(
            "switch_S37728", pr, calls, steps, warmup, peaks,
            what="QKV shape at S=37728, per call: adapter a (rank 384) s=1, b (rank 128) s=0.5, NULL, a s=0, "
                 "b s=1, a s=0.5; FLOPs count the LoRA only where it runs (strength 0 and NULL take the base path)")
        del pr
    sweep = None
    if not a.no_sweep:
        sweep = []
        for M in configs.SWEEP_M:
            x, s, W, ads = futs.pop(f"sweep_M{M}").result()
            pr = Projection(x, s, W, ads, False, device)
            line = projection_line(f"sweep_M{M}", pr, [(0, 1.0)], steps, warmup, peaks,
                                   host=(x, s, W, ads[0], False),
                                   what="QKV 5120->15360 rank 384, Student-t(3) activations with 1% outlier channels")
            tiles = ((M + 255) // 256) * (pr.N // 256)
            line["gemm_tiles"] = tiles
            line["gemm_tile_waves"] = tiles / (torch.cuda.get_device_properties(device).multi_processor_count // 2)
            sweep.append(line)
            del pr
    return out, sweep

# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- CPU oracle
def oracle_sample_run(host, m_rows, n_cols, seed=123, packed=None):
    """Run the oracle on a row x output-column sample of every projection as
    its own call (amax over the sampled rows).  With only a column sample of
    gate/up there is no full SiLU*up row to feed down, so down's sampled rows
    are drawn from N(0, 1) instead.  Returns (seconds, flops)."""
    from oracle import linear
    rng = np.random.default_rng(seed)
    t_total, flops = 0.0, 0
    for i, p in enumerate(host):
        K, N, r, silu = p["K"], p["N"], p["rank"], p["silu"]
        wq, ws, tsw = packed[i] if packed else linear.pack_weight(p["W"])
        if silu:
            half = N // 2
            nc = min(n_cols // 2, half)
            c = np.sort(rng.choice(half, nc, replace=False))
            cols = np.concatenate([c, c + half])
        else:
            nc = min(n_cols, N)
            cols = np.sort(rng.choice(N, nc, replace=False))
        weight = (wq[cols], ws[cols], tsw)
        ad = dict(p["adapter"])
        ad["B"] = ad["B"][cols]
        if p["x"] is not None:
            rows = np.sort(rng.choice(p["x"].shape[0], m_rows, replace=False))
            x = p["x"][rows]
        else:
            x = synth.bf16_round(rng.standard_normal((m_rows, K)).astype(np.float32))
        t0 = time.perf_counter()
        y = linear.forward(x, weight, p["pqs"], ad, 1.0, silu)
        t_total += time.perf_counter() - t0
        flops += 2 * x.shape[0] * (K * len(cols) + K * r + r * len(cols))
    return t_total, flops


def pack_all(host):
    from oracle import linear
    return [linear.pack_weight(p["W"]) for p in host]


def calibrate_sample(host, packed, seconds):
    """Pick (rows, cols) so that one oracle sample run takes about ``seconds``:
    widen the column sample first (up to 4096 output columns), then the rows."""
    S = max(p["x"].shape[0] for p in host if p["x"] is not None)
    m, n = 16, 256
    for _ in range(16):
        t, _ = oracle_sample_run(host, m, n, packed=packed)
        if t >= 0.6 * seconds:
            break
        grow = min(4.0, seconds / max(t, 1e-3))
        if n < 4096:
            n = int(min(4096, n * grow)) // 128 * 128
        elif m < S:
            m = int(min(S, m * grow))
        else:
            break
    return m, n


def cpu_info():
    """Threads the oracle's BLAS calls use (all host cores unless limited)."""
    try:
        from threadpoolctl import threadpool_info
        n = max((d.get("num_threads") or 0) for d in threadpool_info() if d.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# -------------------------------------------------------------------- arms
def reference_arm(a, rank, world):
    if rank != 0:
        return 0
    S = a.S
    host = make_block_inputs(S)
    packed = pack_all(host)
    per_step = 150.0 / max(1, a.steps + a.warmup)
    m, n = calibrate_sample(host, packed, per_step)
    for _ in range(a.warmup):
        oracle_sample_run(host, m, n, packed=packed)
    t_sum, f_sum = 0.0, 0
    for k in range(a.steps):
        t, f = oracle_sample_run(host, m, n, seed=1000 + k, packed=packed)
        t_sum += t
        f_sum += f
    value = f_sum / t_sum / 1e12
    sample = f"{m} rows x {n} output columns of each of the 4 projections per step (S={S} workload)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * t_sum / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"dit_block_4proj_S{S}", "S": S, "hidden": configs.HIDDEN, "mlp": configs.MLP,
                       "ranks": [p[3] for p in configs.BLOCK_PROJECTIONS], "strength": 1.0},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_info(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def fused_qkv_rope_line(blk, wq, wk, pos, c, a, qkv_gemm_ms, rope_ms):
    """The QKV GEMM stage with Q/K RMSNorm + RoPE in its epilogue
    (h3lin_forward_gemm_qk_rope: the angle-table pass + the GEMM) on the
    block's prepared QKV workspace, timed like the plain stage, against that
    stage + the separate in-place pass; its output is checked bit for bit
    against the two-step result on the same inputs."""
    import torch
    h = blk.h3lin
    d = blk.proj[0]
    S = blk.S
    prm = h.rope_params(c["heads"], 128, c["rot"], c["axis_dims"], c["theta"], c["eps"])
    wsb = h.h3lin_forward_qk_rope_workspace_bytes(S, d["K"], d["N"], d["rank"])
    ws = h.new_workspace(wsb)
    out = torch.empty_like(d["out"])
    ref = torch.empty_like(d["out"])
    st = d["stream"]

    def check(code, what):
        if code:
            raise h.H3linError(code, what)

    check(h.h3lin_forward_prepare(d["x_dev"].data_ptr(), S, d["pqs_dev"].data_ptr(), d["wc"], d["ac"], 1.0,
                                  ws.data_ptr(), ws.numel(), st), "h3lin_forward_prepare")

    def fused():
        check(h.h3lin_forward_gemm_qk_rope(S, d["wc"], d["ac"], 1.0, prm, wq.data_ptr(), wk.data_ptr(), pos.data_ptr(),
                                           out.data_ptr(), ws.data_ptr(), ws.numel(), st), "h3lin_forward_gemm_qk_rope")

    for _ in range(max(3, a.warmup)):
        fused()
    n = max(10, a.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        fused()
    e1.record()
    torch.cuda.synchronize()
    fms = e0.elapsed_time(e1) / n
    # the two-step result on the same workspace
    check(h.h3lin_forward_gemm(S, d["wc"], 0, d["ac"], 1.0, ref.data_ptr(), h.H3LIN_OUT_BF16, ws.data_ptr(),
                               ws.numel(), st), "h3lin_forward_gemm")
    h.qk_norm_rope(ref, wq, wk, pos, c["heads"], c["rot"], c["axis_dims"], c["theta"], c["eps"], workspace=ws)
    torch.cuda.synchronize()
    same = bool(torch.equal(out.view(torch.int16), ref.view(torch.int16)))
    if h.read_status(ws) != 0:
        raise RuntimeError("device status set by h3lin_forward_gemm_qk_rope")
    del ws, out, ref
    return {"ms": fms, "launches": 2 * n, "qkv_gemm_ms": qkv_gemm_ms, "qk_norm_rope_ms": rope_ms,
            "two_step_ms": qkv_gemm_ms + rope_ms, "saved_ms": qkv_gemm_ms + rope_ms - fms,
            "bit_identical_to_two_step": same,
            "what": "h3lin_forward_gemm_qk_rope on the block's QKV (angle table + pair GEMM whose epilogue "
                    "normalises and rotates Q and K before the store) vs the plain QKV GEMM + h3lin_qk_norm_rope"}


def native_arm(a, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from nvfp4_linear_lora_gb300 import build as h3build
    h3build.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    S = a.S
    import concurrent.futures as cf
    pool = cf.ThreadPoolExecutor(max_workers=4)
    futs = start_workload_inputs(a, pool) if rank == 0 else {}
    host = make_block_inputs(S)
    blk = Block(host, S, device, fused_mlp=not a.unfused_mlp)
    peaks, peak_kind = load_peaks()
    total, base, ldown, lup = block_flops(S)

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up
    for _ in range(a.warmup):
        blk.step()
    torch.cuda.synchronize()
    blk.check_status()

    # timed region: K steps, GEMM kernels bracketed by events on the launching stream
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in blk.proj]
          for _ in range(a.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local_rank) if rank == 0 else None
    time.sleep(0.3 if clk else 0)
    t0.record()
    for k in range(a.steps):
        blk.step(gemm_events=ev[k])
    t1.record()
    torch.cuda.synchronize()
    clocks = clk.stop() if clk else None
    barrier()
    ms = t0.elapsed_time(t1) / a.steps
    gemm_ms = [statistics.mean(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(a.steps))
               for i in range(len(blk.proj))]
    blk.check_status()
    ms = max_over_ranks(ms, world, device)
    value = whole_job_tflops(total, world, ms)

    # the step after QKV: Q/K RMSNorm + split-half three-axis RoPE, in place on
    # the block's QKV output (1.16 GB, larger than L2), timed alone
    rope_line = None
    if not a.no_rope:
        c = configs.ROPE
        qkv_out = blk.proj[0]["out"]
        rrng = np.random.default_rng(configs.ROPE_SEED)
        wq = torch.from_numpy(synth.norm_gain(rrng, 128)).to(device)
        wk = torch.from_numpy(synth.norm_gain(rrng, 128)).to(device)
        pos = torch.from_numpy(synth.rope_positions(S, c["frames"], c["height"], c["width"])).to(device)
        h3r = blk.h3lin
        ws_r = h3r.new_workspace(h3r.h3lin_quant_workspace_bytes(), device)

        def rope_once():
            h3r.qk_norm_rope(qkv_out, wq, wk, pos, c["heads"], c["rot"], c["axis_dims"], c["theta"], c["eps"],
                             workspace=ws_r)

        for _ in range(max(3, a.warmup)):
            rope_once()
        n_r = max(10, a.steps // 4)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        r0.record()
        for _ in range(n_r):
            rope_once()
        r1.record()
        torch.cuda.synchronize()
        if h3r.read_status(ws_r) != 0:
            raise RuntimeError("device status set by h3lin_qk_norm_rope")
        rms = r0.elapsed_time(r1) / n_r
        rbytes = S * 2 * c["heads"] * 128 * 2 * 2 + S * 12
        rope_line = {"ms": rms, "launches": n_r, "algorithmic_bytes": rbytes,
                     "achieved_gbs": rbytes / (rms * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                     "frac": rbytes / (rms * 1e-3) / 1e9 / peaks["hbm_gbs"], "bound": "hbm",
                     "what": "h3lin_qk_norm_rope in place on the block's QKV output [S, 15360] bf16: per-head "
                             "RMSNorm of Q and K, split-half RoPE of 96 of 128 dims over (t, h, w) positions; "
                             "bytes = Q and K read and written once + positions"}
        rope_line["fused_in_qkv_gemm"] = fused_qkv_rope_line(blk, wq, wk, pos, c, a, gemm_ms[0], rms)

    # the step before QKV: the modulation producer (LayerNorm + segment-wise
    # AdaLN shift/scale -> bf16 LoRA input + amax partials), then QKV's prepare
    # from those partials (one pass over x_mod) against the plain prepare
    mod_line = None
    if not a.no_modulation:
        c = configs.MODULATION
        h3m = blk.h3lin
        mrng = np.random.default_rng(configs.MODULATION_SEED)
        xres = synth.to_bf16_tensor(synth.residual(mrng, S, configs.HIDDEN)).to(device)
        tab = torch.from_numpy(synth.adaln_table(mrng, len(c["segments"]), configs.HIDDEN)).to(device)
        rtab = torch.from_numpy(synth.segment_rows(c["segments"])).to(device)
        q = blk.proj[0]
        xmod = torch.empty_like(xres)

        def mod_once():
            h3m.modulate_produce(xres, tab, rtab, q["ws"], q["pqs_dev"], c["eps"], out=xmod)

        def timed(fn, n):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        n_m = max(10, a.steps // 4)
        mms_ = timed(mod_once, n_m)

        def prep(fn):
            st = fn(xmod.data_ptr(), S, q["pqs_dev"].data_ptr(), q["wc"], q["ac"], 1.0, q["ws"].data_ptr(),
                    q["ws"].numel(), q["stream"])
            if st:
                raise h3m.H3linError(st, "prepare")

        mod_once()
        p_prod = timed(lambda: prep(h3m.h3lin_forward_prepare_produced), n_m)
        p_plain = timed(lambda: prep(h3m.h3lin_forward_prepare), n_m)
        if h3m.read_status(q["ws"]) != 0:
            raise RuntimeError("device status set by the modulation producer")
        mbytes = S * configs.HIDDEN * 4 + S * 4
        mod_line = {"ms": mms_, "launches": n_m, "algorithmic_bytes": mbytes,
                    "achieved_gbs": mbytes / (mms_ * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                    "frac": mbytes / (mms_ * 1e-3) / 1e9 / peaks["hbm_gbs"], "bound": "hbm",
                    "qkv_prepare_from_partials_ms": p_prod, "qkv_prepare_plain_ms": p_plain,
                    "what": "h3lin_modulate_produce on the block's QKV input [S, 5120]: LayerNorm + (1 + scale) "
                            "and shift gathered from a 3-row AdaLN table by segment, bf16 out, amax partials for "
                            "QKV; bytes = x read + x_mod written once. Then QKV's prepare from those partials "
                            "(one pass over x_mod: quantise + A(x)) vs the plain prepare (amax pass + quantise)"}

    # merged-LoRA comparison mode: each weight with its adapter folded in
    # (h3lin_merge_lora), re-packed, then the block on the base path only
    merged_line = None
    if not a.no_merged:
        h3 = blk.h3lin
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        packed_m = []
        merge_ms = 0.0
        for p, d in zip(host, blk.proj):
            Wd = synth.to_bf16_tensor(p["W"]).to(device)
            m0.record()
            h3.merge_lora(Wd, d["ad"], 1.0, d["pqs_dev"], out=Wd)
            pwm = h3.pack_weight(Wd)
            m1.record()
            torch.cuda.synchronize()
            merge_ms += m0.elapsed_time(m1)
            del Wd
            packed_m.append(pwm)
        saved = [(d["wc"], d["ac"]) for d in blk.proj]
        for d, pwm in zip(blk.proj, packed_m):
            d["wc"], d["ac"] = pwm.c_struct(), None
        try:
            for _ in range(a.warmup):
                blk.step()
            torch.cuda.synchronize()
            n_m = max(10, a.steps // 4)
            barrier()
            torch.cuda.synchronize()
            t0.record()
            for _ in range(n_m):
                blk.step()
            t1.record()
            torch.cuda.synchronize()
            barrier()
            mms = t0.elapsed_time(t1) / n_m
            blk.check_status()
        finally:
            for d, (wc, ac) in zip(blk.proj, saved):
                d["wc"], d["ac"] = wc, ac
        mms = max_over_ranks(mms, world, device)
        merged_line = {"ms_per_block": mms, "steps": n_m,
                       "base_tflops": world * base / (mms * 1e-3) / 1e12,
                       "dynamic_over_merged_time": ms / mms,
                       "merge_and_pack_ms": merge_ms,
                       "what": "adapter folded into each weight (h3lin_merge_lora, strength 1) and re-packed; "
                               "the block then runs the base path only (adapter NULL). A speed bound for the "
                               "dynamic path, paid for by re-packing per adapter/strength switch"}

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if not a.no_e2e:
        # End to end through the C ABI: every step copies its three activations
        # from pinned host memory and reads its three block outputs back.  The
        # copies of neighbouring steps run on their own streams, overlapped with
        # the block compute (double-buffered device inputs and outputs); the
        # timed region spans the first step's H2D to the last step's D2H.
        xs_host = [synth.to_bf16_tensor(p["x"]).pin_memory() for p in host if p["x"] is not None]
        outs0 = [blk.proj[0]["out"], blk.proj[1]["out"], blk.proj[3]["out"]]
        x_slots = [[d["x_dev"] for d in blk.proj[:3]], [torch.empty_like(d["x_dev"]) for d in blk.proj[:3]]]
        out_slots = [outs0, [torch.empty_like(o) for o in outs0]]
        outs_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs0]
        h2d = sum(t.numel() * t.element_size() for t in xs_host)
        d2h = sum(t.numel() * t.element_size() for t in outs_host)
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def pipelined(n):
            for i in range(n):
                sl = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp_done[sl])        # slot sl's inputs were read by step i - 2
                    for hsrc, ddst in zip(xs_host, x_slots[sl]):
                        ddst.copy_(hsrc, non_blocking=True)
                    in_done[sl].record(s_in)
                comp.wait_event(in_done[sl])
                if i >= 2:
                    comp.wait_event(out_done[sl])             # slot sl's outputs were read back by step i - 2
                blk.step_io(x_slots[sl], out_slots[sl])
                comp_done[sl].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[sl])
                    for dsrc, hdst in zip(out_slots[sl], outs_host):
                        hdst.copy_(dsrc, non_blocking=True)
                    out_done[sl].record(s_out)
            comp.wait_event(out_done[(n - 1) % 2])

        pipelined(max(3, a.warmup // 2))                     # untimed warm-up of the copy path
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0.record(comp)
        s_in.wait_event(e0)
        pipelined(a.e2e_steps)
        e1.record(comp)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1) / a.e2e_steps
        ems = max_over_ranks(ems, world, device)
        blk.check_status()
        e2e = {"value": world * total / (ems * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "H2D of step i+1 and D2H of step i-1 on their own streams, overlapped with step i's "
                          "compute (double-buffered device inputs and outputs)"}

    if rank != 0:
        pool.shutdown(wait=False)
        return 0

    # the single-projection workloads and the sweep (their inputs were drawn
    # on worker threads meanwhile; all drawn before the CPU baseline is timed)
    workloads, sweep = workload_lines(a, device, peaks, futs)
    pool.shutdown(wait=True)

    # roofline of the dominant kernel (the FP4 GEMM with LoRA-up), live event
    # timing; peaks are the burst figures (the timed region is about a second,
    # not a seconds-long power-capped loop)
    gemm_total_ms = sum(gemm_ms)
    peak_bf16 = peaks["bf16_tflops"]
    peak_fp4 = peak_bf16 * FP4_OVER_BF16
    rf = gemm_roofline(base, lup, gemm_total_ms, peaks)
    alg = gemm_algorithmic_bytes(S)
    traffic = None
    if GEMM_TRAFFIC["sources_sha256"] == gemm_sources_sha256() and GEMM_TRAFFIC["S"] == S:
        traffic = sum(GEMM_TRAFFIC["bytes_per_launch"].values())
    roofline = {"kernel": "k_fp4gemm", "bound": "tensor", **rf, "traffic": traffic,
                "traffic_scope": "DRAM bytes of the block's four GEMM launches (read + write), as achieved is "
                                 "the FLOPs of those four launches over their summed time",
                "algorithmic_bytes": sum(alg.values()),
                "traffic_per_launch": dict(GEMM_TRAFFIC["bytes_per_launch"]) if traffic else None,
                "peak_basis": f"{peak_kind} burst bf16 {peak_bf16:.1f} TF/s x {FP4_OVER_BF16:g} for the FP4 part "
                              f"(FP4 {peak_fp4:.0f} TF/s), x 1 for the BF16 LoRA-up part, time-weighted over this "
                              f"kernel's FLOP mix",
                "gemm_ms_per_projection": dict(zip([d["name"] for d in blk.proj], gemm_ms))}

    cpu = None
    if not a.no_cpu_baseline and world == 1:
        packed = pack_all(host)
        m, n = calibrate_sample(host, packed, a.cpu_seconds)
        t, f = oracle_sample_run(host, m, n, seed=7, packed=packed)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cpu_info(), "kind": "oracle",
               "sample": f"{m} rows x {n} output columns of each projection (same S={S} workload), {t:.1f} s"}

    # the base-only fraction of the FP4 peak and the BF16-peak fraction of the
    # LoRA part: the merged-LoRA block does the same base work with no LoRA
    # branch, and the dynamic block's extra time is what its A(x) and B(u) cost
    split = None
    if merged_line is not None:
        mms = merged_line["ms_per_block"]
        lora_ms = ms - mms
        split = {"base_only": {"ms_per_block": mms, "tflops": world * base / (mms * 1e-3) / 1e12,
                               "frac_of_fp4_peak": base / (mms * 1e-3) / 1e12 / peak_fp4},
                 "lora_part": {"ms_per_block": lora_ms,
                               "marginal_tflops": None if lora_ms <= 0 else (ldown + lup) / (lora_ms * 1e-3) / 1e12},
                 "how": "base only = the block with every adapter merged into its weight (merged_lora: the same "
                        "base work, no LoRA branch); LoRA part = the dynamic block's extra time over it, for the "
                        "A(x) and B(u) FLOPs: a marginal time (A(x) runs inside the HBM-bound amax pass, where it "
                        "partly hides), not a kernel's fraction of a peak"}


    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e2m1+bf16", "data": "synthetic",
            "config": {"workload": f"dit_block_4proj_S{S}", "S": S, "hidden": configs.HIDDEN, "mlp": configs.MLP,
                       "ranks": [p[3] for p in configs.BLOCK_PROJECTIONS], "strength": 1.0,
                       "mlp_path": "producer-fused (gate/up epilogue reduces amax(h*s) for down)" if blk.fused_mlp
                                   else "unfused (separate amax pass over h)",
                       "l2": f"inputs larger than L2 (each activation >= {S * configs.HIDDEN * 2 / 1e6:.0f} MB), no flush"},
            "ms_per_block": ms, "frac_of_fp4_peak": value / world / peak_fp4,
            "frac_of_fp4_nominal": value / world / FP4_NOMINAL_TFLOPS,
            "fp4_peak_basis": f"frac_of_fp4_peak: {peak_kind} burst bf16 {peak_bf16:.1f} TF/s x {FP4_OVER_BF16:g} = "
                              f"{peak_fp4:.0f} TF/s; frac_of_fp4_nominal: datasheet dense FP4 {FP4_NOMINAL_TFLOPS:.0f} "
                              f"TF/s; SM clock median in the timed region: "
                              f"{clocks.get('sm_mhz') if clocks else None} MHz",
            "flops_per_block": {"total": total, "base_fp4": base, "lora_down": ldown, "lora_up": lup},
            "kernel_ms": {"gemm": gemm_total_ms, "prepare": ms - gemm_total_ms},
            "roofline": roofline, "peak_split": split, "cpu_baseline": cpu, "e2e": e2e, "merged_lora": merged_line,
            "qk_norm_rope": rope_line, "modulation": mod_line,
            "configs": workloads, "sweep": sweep,
            "gpu_launches": blk.launches_per_step() * a.steps, "clocks": clocks,
            "peaks": {"kind": peak_kind, **peaks}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    a = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", a.gpus if a.gpus == 1 else 1))
    rank = int(os.environ.get("RANK", 0))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1 and a.impl == "native":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if a.impl == "reference":
            return reference_arm(a, rank, world)
        return native_arm(a, rank, world, local_rank)
    finally:
        if world > 1 and a.impl == "native":
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
