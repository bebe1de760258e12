#!/usr/bin/env python3
"""Benchmark of the NVFP4 W4A4 Gated DeltaNet layer step on GB300.

Headline workload: the full-width layer (hidden 2048, 16 key / 32 value heads,
d 128, conv 4, NVFP4 weights) in decode bucket c1, replayed as a CUDA graph.
One bench step = one decode step through a stack of L distinct layer
instances (own weights and state each) whose footprint is > 4x the L2 cache,
so every layer-step streams its weights and state from HBM. The reported value
is microseconds per layer-step (lower is better).

Also reported: buckets c2..c16, batch 256 and prefill tokens/s (extra keys),
the roofline of the dominant kernel (the W4A4 projection GEMV), an
end-to-end leg through the Python API with host buffers, SM clocks sampled
during the timed region, and the CPU oracle timed on a bounded sample.

--impl reference times the CPU oracle on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN layer decode us/step at c1..c16 & prefill tok/s; HBM GB/s vs GB300 peak"
UNIT = "us/step"

# Algorithmic bytes of one decode layer-step: weights once + per active sequence.
W_BYTES = 14_155_776 + 73_728 + 4_718_592 + 65_536 + 256 + 512      # 19,014,400
SEQ_BYTES = 4_194_304 + 98_304 + 4_096 + 4_096                       # 4,300,800
GEMV_IN_BYTES = 12352 * (1024 + 128)                                  # qkvz+ba codes+scales


def layer_bytes(sh, state_bf16=False):
    """(weight bytes, bytes per active sequence) of one decode layer-step of shape sh:
    NVFP4 codes + E4M3 scales of the three projections, conv taps (BF16), A_log and
    dt_bias, the norm weight; per sequence the FP32 state and BF16 conv state read
    and written, x in and out."""
    nvfp4 = lambda rows, k: rows * (k // 2 + k // 16)
    w = (nvfp4(sh.qkvz_out, sh.hidden) + nvfp4(sh.ba_out, sh.hidden) + nvfp4(sh.hidden, sh.value_dim)
         + sh.conv_channels * sh.conv_kernel * 2 + sh.n_v_heads * 8 + sh.d_v * 4)
    seq = (2 * sh.n_v_heads * sh.d_v * sh.d_k * (2 if state_bf16 else 4) + 2 * (sh.conv_kernel - 1) * sh.conv_channels * 2
           + 2 * sh.hidden * 2)
    return w, seq


def step_bytes(B: int, sh=None, state_bf16=False) -> int:
    if sh is None and not state_bf16:
        return W_BYTES + B * SEQ_BYTES
    from nvfp4_gated_deltanet_gb300 import synth
    w, seq = layer_bytes(sh or synth.FULL, state_bf16)
    return w + B * seq


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi SM clock / throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload

def make_stack(pkg, synth, n_layers, B, max_batch, device="cuda", shape=None, state_bf16=False):
    """n_layers layer contexts sharing one synthetic weight set (uploaded once
    per context, so each has its own copy in HBM), each with B slots of state."""
    import numpy as np
    import torch
    sh = shape or synth.FULL
    w = synth.layer_weights(sh, 1)
    layers, states = [], []
    conv0 = np.stack([synth.conv_state(sh, synth.slot_seed(s)) for s in range(B)])
    ssm0 = np.stack([synth.ssm_state(sh, synth.slot_seed(s)) for s in range(B)])
    x = np.stack([synth.x_tokens(sh, synth.slot_seed(s), 1)[0] for s in range(B)])
    xd = torch.from_numpy(x.view(np.int16)).to(device)
    for _ in range(n_layers):
        L = pkg.layer_from_synth(w, max_batch=max_batch, state_bf16=state_bf16)
        layers.append(L)
        ssm = torch.from_numpy(ssm0).to(device)
        if state_bf16:   # the same values stored as BF16 bits (round to nearest even)
            ssm = ssm.to(torch.bfloat16).view(torch.int16)
        states.append((torch.from_numpy(conv0.view(np.int16)).to(device), ssm))
    return w, layers, states, xd


def capture_stack(layers, states, xd, B):
    import torch
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    outs = [torch.empty(B, layers[0].H, dtype=torch.int16, device="cuda") for _ in layers]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for L, (c, m), o in zip(layers, states, outs):
            L.decode_step(xd[:B], ids, c, m, out=o)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for L, (c, m), o in zip(layers, states, outs):
            L.decode_step(xd[:B], ids, c, m, out=o)
    torch.cuda.synchronize()
    return g, outs


def time_graph(g, steps, warmup):
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps  # ms per bench step


# Algorithmic bytes per launch of the c1 step's three kernels as the roofline leg
# runs them (full-width layer, one row): the in-projection reads its weights
# (q|k|v|z|b|a codes + scales) and x, writes the BF16 projections; the mixing
# stage (gdn_mix_step) reads the projections, conv taps, gate parameters and
# norm weight, reads and writes the FP32 recurrent state and the conv state,
# writes y in FP32; the out-projection reads its weights and y (NVFP4), writes out.
STAGE_KERNELS = {
    "in_proj": "gemv_mma_kernel<2,4> (one-row W4A4 q|k|v|z|b|a projection, warp-MMA block products)",
    "mix": "mix_kernel<128,4> (conv, norms, gates, gated delta rule, gated RMSNorm, NVFP4 y)",
    "out_proj": "gemv_mma_kernel<1,8> (one-row W4A4 out-projection)",
}
# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture of
# the current kernels (profiles/decode_c1_inproj_mix_ncu.md); a stage absent
# here has no capture of its current form
STAGE_TRAFFIC = {"in_proj": 14_252_544, "mix": 2_278_912}
STAGE_BYTES = {
    "in_proj": GEMV_IN_BYTES + 2048 * 2 + 12352 * 2,
    "mix": 12352 * 2 + 8192 * 4 * 2 + 32 * 8 + 128 * 4 + 2 * 2_097_152 + 2 * 3 * 8192 * 2 + 4096 * 4,
    "out_proj": 2048 * (2048 + 256) + 2048 + 256 + 2048 * 2,
}


def time_stages(pkg, layers, states, xd, steps):
    """The c1 step's three kernels one at a time over the stack's layer
    instances (each launch on its own layer's weights and state), each as one
    CUDA graph timed with CUDA events on its stream: us per launch."""
    import torch
    L0 = layers[0]
    x1 = xd[:1].contiguous()
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    nin = 2 * L0.Hk * L0.D + 2 * L0.Hv * L0.D + 2 * L0.Hv
    proj = [torch.empty(1, nin, dtype=torch.int16, device="cuda") for _ in layers]
    ycs = [torch.empty(1, L0.Hv * L0.D // 2, dtype=torch.uint8, device="cuda") for _ in layers]
    yss = [torch.empty(1, L0.Hv * L0.D // 16, dtype=torch.uint8, device="cuda") for _ in layers]
    yf = torch.empty(1, L0.Hv * L0.D, dtype=torch.float32, device="cuda")
    out = torch.empty(1, L0.H, dtype=torch.int16, device="cuda")
    for i, L in enumerate(layers):  # real projections and y for the later stages
        L.in_proj(x1, None, proj[i])
        ycs[i].zero_()
        yss[i].fill_(0x38)
    torch.cuda.synchronize()
    nq = 2 * L0.Hk * L0.D + 2 * L0.Hv * L0.D
    passes = {
        "in_proj": lambda: [L.in_proj(x1, None, proj[i]) for i, L in enumerate(layers)],
        "mix": lambda: [L.mix_step(proj[i][:, :nq], proj[i][:, nq:], ids, c, m, y=yf)
                        for i, (L, (c, m)) in enumerate(zip(layers, states))],
        "out_proj": lambda: [L.out_proj(ycs[i], yss[i], out=out) for i, L in enumerate(layers)],
    }
    res = {}
    for name, fn in passes.items():
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        res[name] = time_graph(g, steps, 3) / len(layers) * 1e3
        del g
    return res


def time_batch(pkg, synth, B, hbm_peak, n_layers=2, steps=10, state_bf16=False):
    """Large-batch decode: B sequences per step through n_layers layer instances
    (each layer-step moves > 300 MB, far beyond L2)."""
    w, layers, states, xd = make_stack_b(pkg, synth, n_layers, B, state_bf16=state_bf16)
    g, _ = capture_stack(layers, states, xd, B)
    ms = time_graph(g, steps, 3)
    us = ms * 1e3 / n_layers
    gbs = step_bytes(B, state_bf16=state_bf16) / (us * 1e-6) / 1e9
    return {"us_per_layer_step": round(us, 2), "tokens_per_s": round(B / (us * 1e-6)), "hbm_gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / hbm_peak, 4)}


def make_stack_b(pkg, synth, n_layers, B, device="cuda", state_bf16=False):
    import numpy as np
    import torch
    w = synth.layer_weights(synth.FULL, 1)
    x = np.stack([synth.x_tokens(synth.FULL, synth.slot_seed(s), 1)[0] for s in range(B)])
    xd = torch.from_numpy(x.view(np.int16)).to(device)
    layers, states = [], []
    for _ in range(n_layers):
        L = pkg.layer_from_synth(w, max_batch=B, state_bf16=state_bf16)
        conv = torch.empty(B, 3, synth.FULL.conv_channels, dtype=torch.int16, device=device)
        ssm = torch.empty(B, synth.FULL.n_v_heads, 128, 128, dtype=torch.float32, device=device)
        conv.copy_(torch.from_numpy(synth.conv_state(synth.FULL, 100).view(np.int16)).to(device).expand_as(conv))
        ssm.copy_(torch.from_numpy(synth.ssm_state(synth.FULL, 100)).to(device).expand_as(ssm))
        if state_bf16:
            ssm = ssm.to(torch.bfloat16).view(torch.int16)
        layers.append(L)
        states.append((conv, ssm))
    return w, layers, states, xd


def time_verify(layers, states, xd, B, r, steps):
    """Verify of r candidate tokens for B sequences, then the commit of every
    token, per layer instance of the stack, as one CUDA graph; us per layer."""
    import torch
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), r, dtype=torch.int32, device="cuda")
    x = xd[:B].unsqueeze(1).expand(B, r, -1).contiguous()
    snaps = [L.new_snapshots(B, r) for L in layers]
    outs = [torch.empty(B, r, layers[0].H, dtype=torch.int16, device="cuda") for _ in layers]

    def one_pass():
        for L, (c, m), (sc, ss), o in zip(layers, states, snaps, outs):
            L.verify(x, ids, c, m, sc, ss, out=o)
            L.verify_commit(ids, acc, sc, ss, c, m)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        one_pass()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        one_pass()
    us = time_graph(g, steps, 3) * 1e3 / len(layers)
    del g, snaps
    return {"us_per_layer": round(us, 3), "tokens_per_s": round(B * r / (us * 1e-6)),
            "note": f"{B} sequences x {r} candidate tokens, verify + commit of all"}


def time_kda(pkg, synth, M, H, D, state_bf16, hbm_peak, l2, steps):
    """KDA-style recurrent step for M streams x H heads: a graph of n steps over
    n distinct state buffers (n x state bytes > 4x L2); us per layer-step and
    GB/s of algorithmic bytes (state read + write, q/k/v/g/beta in, o out)."""
    import torch
    q, k, v, g, beta, S = synth.kda_inputs(M, H, D, 5)
    dev = lambda a: torch.from_numpy(a).cuda()
    q, k, v, g, beta = dev(q), dev(k), dev(v), dev(g), dev(beta)
    es = 2 if state_bf16 else 4
    sbytes = M * H * D * D * es
    n = min(256, max(4, -(-4 * l2 // sbytes) + 1))
    S0 = dev(S)
    if state_bf16:
        S0 = S0.to(torch.bfloat16).view(torch.int16)
    states = [S0.clone() for _ in range(n)]
    o = torch.empty(M, H, D, dtype=torch.float32, device="cuda")

    def one_pass():
        for st in states:
            pkg.kda_step(q, k, v, g, beta, st, o=o)
    one_pass()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        one_pass()
    us = time_graph(gr, steps, 3) * 1e3 / n
    nbytes = 2 * sbytes + (5 * M * H * D + M * H) * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    del gr, states
    return {"us_per_layer_step": round(us, 3), "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / hbm_peak, 4),
            "layers": n, "state": "bf16" if state_bf16 else "f32", "shape": f"M{M} H{H} d{D}"}


def time_prefill(pkg, synth, T, reps=3):
    """Prefill of one T-token sequence from zero state (weights stay resident
    in L2 within the call, as they would in a real prompt)."""
    import numpy as np
    import torch
    w = synth.layer_weights(synth.FULL, 1)
    L = pkg.layer_from_synth(w, max_batch=1, max_prefill_tokens=T)
    x = torch.from_numpy(synth.x_tokens(synth.FULL, 7, T).view(np.int16)).cuda()
    conv, ssm = L.new_states(1)
    out = torch.empty(T, synth.FULL.hidden, dtype=torch.int16, device="cuda")
    L.prefill(x, 0, True, conv, ssm, out=out)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        L.prefill(x, 0, True, conv, ssm, out=out)
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    return {"ms": round(ms, 3), "tokens_per_s": round(T / (ms * 1e-3))}


def max_over_ranks(x: float, dist=None) -> float:
    """The largest x over all ranks (every rank gets it); x itself without a
    process group. NCCL reduces a device tensor, other backends a host one."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def fp4_peak():
    """Dense FP4 tensor peak: the measured BF16 GEMM burst x the nominal FP4 / BF16
    ratio (13.5 / 2.25 PFLOP/s dense)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]) * 6.0, "measured bf16 burst x 6 (nominal fp4/bf16 ratio)"
    except Exception:
        return 1900.0 * 6.0, "fallback bf16 x 6 (nominal fp4/bf16 ratio)"


def time_in_proj(pkg, synth, T, reps=20):
    """The prefill in-projection alone (NVFP4 quantisation of x, then the W4A4
    q|k|v|z|b|a GEMM on tcgen05) over T tokens, through gdn_in_proj."""
    import numpy as np
    import torch
    w = synth.layer_weights(synth.FULL, 1)
    L = pkg.layer_from_synth(w, max_batch=1, max_prefill_tokens=T)
    x = torch.from_numpy(synth.x_tokens(synth.FULL, 7, T).view(np.int16)).cuda()
    nin = 2 * L.Hk * L.D + 2 * L.Hv * L.D + 2 * L.Hv
    out = torch.empty(T, nin, dtype=torch.int16, device="cuda")
    for _ in range(3):
        L.in_proj(x, None, out)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        L.in_proj(x, None, out)
    e1.record(st)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    tflops = 2.0 * nin * T * L.H / (us * 1e-6) / 1e12
    peak, kind = fp4_peak()
    return {"us": round(us, 2), "tflops": round(tflops, 1), "fp4_peak_tflops": round(peak, 1),
            "frac_of_fp4_peak": round(tflops / peak, 4), "peak_kind": kind,
            "note": "quantisation kernel + persistent tcgen05 GEMM; operands L2-resident"}


def cpu_baseline_leg(seconds_budget=15.0):
    """The oracle, single-threaded, on config-1 decode steps: a bounded sample."""
    code = (
        "import os,sys,time,json;sys.path.insert(0,%r);"
        "from nvfp4_gated_deltanet_gb300 import synth;from oracle import gdn;import numpy as np;"
        "w=synth.layer_weights(synth.FULL,1);L=gdn.Layer(w);x=synth.x_tokens(synth.FULL,101,1000);"
        "c=synth.conv_state(synth.FULL,101)[None].copy();s=synth.ssm_state(synth.FULL,101)[None].copy();"
        "L.decode_step(x[0:1],[0],c,s);t=time.time();n=0\n"
        "while time.time()-t<%f and n<999:\n n+=1;L.decode_step(x[n:n+1],[0],c,s)\n"
        "print(json.dumps({'n':n,'s':time.time()-t}))" % (ROOT, seconds_budget))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["s"] / d["n"] * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{d['n']} config-1 decode c1 layer-steps (full width), single thread, float64/int64 exact"}


def cpu_all_cores_leg(seconds_budget=10.0):
    """The oracle on every host core: one single-threaded process per core, each
    running config-1 decode steps of its own sequence for the same window;
    aggregate throughput as us per layer-step. Workers are capped by the host
    memory (about 2 GB each while the oracle layer is built)."""
    cores = os.cpu_count() or 1
    try:
        with open("/proc/meminfo") as f:
            avail_kb = next(int(ln.split()[1]) for ln in f if ln.startswith("MemAvailable"))
        cores = max(1, min(cores, avail_kb // (2 * 1024 * 1024)))
    except Exception:
        pass
    start_at = time.time() + 20.0  # every worker builds its layer first, then all measure together
    code = (
        "import os,sys,time,json;sys.path.insert(0,%r);"
        "from nvfp4_gated_deltanet_gb300 import synth;from oracle import gdn;import numpy as np;"
        "seed=int(sys.argv[1]);w=synth.layer_weights(synth.FULL,1);L=gdn.Layer(w);"
        "x=synth.x_tokens(synth.FULL,seed,1000);"
        "c=synth.conv_state(synth.FULL,seed)[None].copy();s=synth.ssm_state(synth.FULL,seed)[None].copy();"
        "L.decode_step(x[0:1],[0],c,s)\n"
        "while time.time()<%f: time.sleep(0.01)\n"
        "t=time.time();n=0\n"
        "while time.time()-t<%f and n<999:\n n+=1;L.decode_step(x[n:n+1],[0],c,s)\n"
        "print(json.dumps({'n':n,'t0':t,'t1':time.time()}))" % (ROOT, start_at, seconds_budget))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = [subprocess.Popen([sys.executable, "-c", code, str(100 + i)], stdout=subprocess.PIPE,
                              stderr=subprocess.DEVNULL, text=True, env=env) for i in range(cores)]
    res = []
    for p in procs:
        out, _ = p.communicate(timeout=600)
        if p.returncode == 0 and out.strip():
            res.append(json.loads(out.strip().splitlines()[-1]))
    if not res:
        return None
    n = sum(d["n"] for d in res)
    wall = max(d["t1"] for d in res) - min(d["t0"] for d in res)
    return {"value": wall / n * 1e6, "unit": UNIT, "cores": len(res), "kind": "oracle",
            "sample": f"{n} config-1 decode c1 layer-steps over {len(res)} single-threaded processes "
                      f"(one sequence each) in a {wall:.1f} s window; aggregate throughput"}


def headline_config(world: int) -> dict:
    """The workload of the headline line, identical in both arms."""
    return {"workload": "gdn-decode-c1", "hidden": 2048, "k_heads": 16, "v_heads": 32, "d": 128, "conv": 4,
            "batch": 1, "l2_defeat": "distinct layer instances, footprint > 4x L2",
            "graph": "one CUDA graph per bucket over the stack", "parallelism": f"replicas x{world}"}


def cpu_model() -> str:
    """The host CPU's model string (x86 'model name', else lscpu's 'Model name')."""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


_CPU_SINGLE = r"""
import json, sys, time
sys.path.insert(0, %r)
import numpy as np
from nvfp4_gated_deltanet_gb300 import synth
from oracle import gdn
sh = synth.FULL
w = synth.layer_weights(sh, 1)
L = gdn.Layer(w)
res = {}
def decode(B, steps):
    x = np.stack([synth.x_tokens(sh, synth.slot_seed(s), steps) for s in range(B)], axis=1)
    c = np.stack([synth.conv_state(sh, synth.slot_seed(s)) for s in range(B)])
    m = np.stack([synth.ssm_state(sh, synth.slot_seed(s)) for s in range(B)])
    t = time.perf_counter()
    for i in range(steps):
        L.decode_step(x[i], list(range(B)), c, m)
    return (time.perf_counter() - t) / steps
for B, steps in ((1, 3), (2, 1), (4, 1), (8, 1), (16, 1), (64, 1)):
    res["c%%d" %% B if B <= 16 else "batch%%d" %% B] = {"value": decode(B, steps) * 1e6, "unit": "us/step",
                                                     "sample": "%%d step(s)" %% steps}
T = 64
x = synth.x_tokens(sh, 7, T)
c, m = synth.conv_state(sh, 7, True), synth.ssm_state(sh, 7, True)
t = time.perf_counter()
L.prefill(x, c, m, init_zero=True)
el = time.perf_counter() - t
res["prefill"] = {"value": T / el, "unit": "tokens/s", "sample": "the first %%d tokens of the 1024-token prompt "
                  "(token-by-token recurrence: the cost per token does not depend on T)" %% T}
print(json.dumps(res))
"""


def cpu_configs_leg():
    """The oracle on the host cores for every configuration: single-threaded
    (one process, BLAS pinned to one thread) on a few steps of each decode
    bucket and batch 64 and on a prefill sample; on all cores (oracle.parallel:
    worker processes over rows or key-head groups, bit-identical to the
    single-thread oracle) on one step of c16 and batch 64/128/256 and on whole
    prefills of 1024/4096/16384 tokens. Workers are warmed (weights built)
    before anything is timed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", _CPU_SINGLE % ROOT], capture_output=True, text=True, env=env,
                       timeout=900)
    single = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-300:]}
    import numpy as np
    from nvfp4_gated_deltanet_gb300 import synth
    from oracle import parallel
    sh = synth.FULL
    w = synth.layer_weights(sh, 1)
    pool, n = parallel.make_pool(w)
    allc = {}
    try:
        x1 = synth.x_tokens(sh, 7, 64)
        parallel.prefill(w, x1, synth.conv_state(sh, 7, True), synth.ssm_state(sh, 7, True), True, n, pool)
        for B in (16, 64, 128, 256):
            x = np.stack([synth.x_tokens(sh, synth.slot_seed(s), 1)[0] for s in range(B)])
            c = np.stack([synth.conv_state(sh, synth.slot_seed(s)) for s in range(B)])
            m = np.stack([synth.ssm_state(sh, synth.slot_seed(s)) for s in range(B)])
            t = time.perf_counter()
            parallel.decode_step(w, x, list(range(B)), c, m, n, pool)
            allc["c16" if B == 16 else f"batch{B}"] = {"value": (time.perf_counter() - t) * 1e6, "unit": "us/step",
                                                      "sample": "1 step"}
        for T in (1024, 4096, 16384):
            x = synth.x_tokens(sh, 7, T)
            t = time.perf_counter()
            parallel.prefill(w, x, synth.conv_state(sh, 7, True), synth.ssm_state(sh, 7, True), True, n, pool)
            allc[f"prefill{T}"] = {"value": T / (time.perf_counter() - t), "unit": "tokens/s",
                                   "sample": f"the whole {T}-token prompt"}
    finally:
        pool.close()
        pool.join()
    return {"single_thread": single, "all_cores": allc, "cores_all": n, "cpu_model": cpu_model(),
            "nproc": os.cpu_count()}


def reference_arm(args):
    """--impl reference: the CPU oracle on the same workload and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # one host thread, stated as such (numpy's BLAS would otherwise pick its own)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import numpy as np
    from nvfp4_gated_deltanet_gb300 import synth
    from oracle import gdn
    w = synth.layer_weights(synth.FULL, 1)
    L = gdn.Layer(w)
    x = synth.x_tokens(synth.FULL, 101, args.steps + args.warmup + 1)
    c = synth.conv_state(synth.FULL, 101)[None].copy()
    s = synth.ssm_state(synth.FULL, 101)[None].copy()
    for i in range(args.warmup):
        L.decode_step(x[i:i + 1], [0], c, s)
    t = time.time()
    for i in range(args.steps):
        L.decode_step(x[args.warmup + i:args.warmup + i + 1], [0], c, s)
    el = time.time() - t
    us = el / args.steps * 1e6
    cores = 1
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(args.gpus),
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} config-1 decode c1 layer-steps"},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def single_case(args):
    """One workload alone (prefill of T tokens, or one large-batch decode
    layer-step), for profiling runs: a JSON line with its time."""
    import torch
    import nvfp4_gated_deltanet_gb300 as pkg
    from nvfp4_gated_deltanet_gb300 import synth
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    hbm_peak, _ = peaks()
    if args.case == "prefill":
        r = time_prefill(pkg, synth, args.T, reps=args.steps)
        line = {"case": f"prefill{args.T}", **r}
    elif args.case == "bucket":
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        B = args.batch
        sh = synth.TP2 if args.shape == "tp2" else synth.FULL
        n_layers = args.layers or max(4, -(-4 * l2 // step_bytes(B, sh)) + 1)
        _, layers, states, xd = make_stack(pkg, synth, n_layers, B, max(16, B), shape=sh)
        g, _ = capture_stack(layers, states, xd, B)
        us = time_graph(g, args.steps, args.warmup) * 1e3 / n_layers
        gbs = step_bytes(B, sh) / (us * 1e-6) / 1e9
        line = {"case": f"{'tp2_' if args.shape == 'tp2' else ''}c{B}", "us_per_layer_step": round(us, 3),
                "hbm_gbs": round(gbs, 1),
                "frac_of_peak": round(gbs / hbm_peak, 4), "layers": n_layers}
    else:
        r = time_batch(pkg, synth, args.batch, hbm_peak, steps=args.steps)
        line = {"case": f"batch{args.batch}", **r}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="layer instances in the stack (0: > 4x L2)")
    ap.add_argument("--no-extra", action="store_true", help="skip the c2..c16 / batch / prefill extras")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--case", default="decode", choices=["decode", "prefill", "batch", "bucket"],
                    help="decode: the headline (default); prefill / batch / bucket (a decode stack at --batch "
                         "rows): only that workload, one JSON line (for profiling)")
    ap.add_argument("--T", type=int, default=4096, help="prompt length for --case prefill")
    ap.add_argument("--batch", type=int, default=256, help="rows for --case batch / bucket")
    ap.add_argument("--shape", default="full", choices=["full", "tp2"], help="layer shape for --case bucket")
    ap.add_argument("--tune", default="", help="tuning knobs of gdn_set_tuning to set first, e.g. 13=1,0=1")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.tune and args.impl != "reference":
        import nvfp4_gated_deltanet_gb300 as pkg
        for kv in args.tune.split(","):
            k, v = (int(t) for t in kv.split("="))
            if pkg.lib().gdn_set_tuning(k, v) != 0:
                raise SystemExit(f"bad tuning knob {kv}")
    if args.impl == "reference":
        return reference_arm(args)
    if args.case != "decode":
        return single_case(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import nvfp4_gated_deltanet_gb300 as pkg
    from nvfp4_gated_deltanet_gb300 import synth
    pkg.lib()

    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    per_layer = step_bytes(1)
    n_layers = args.layers or max(4, -(-4 * l2 // per_layer) + 1)
    w, layers, states, xd = make_stack(pkg, synth, n_layers, 16, 16)

    # ---- headline: c1 through the stack
    g1, _ = capture_stack(layers, states, xd, 1)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = time_graph(g1, args.steps, args.warmup)
    ms = max_over_ranks(ms, dist)
    us_layer = ms * 1e3 / n_layers
    hbm_peak, peak_kind = peaks()
    gbs_step = step_bytes(1) / (us_layer * 1e-6) / 1e9

    # ---- the step's kernels one at a time, live: the dominant one by time
    stages = time_stages(pkg, layers, states, xd, max(20, args.steps // 4))
    kernels = {}
    for name, us in stages.items():
        gbs = STAGE_BYTES[name] / (us * 1e-6) / 1e9
        kernels[name] = {"us_per_launch": round(us, 3), "bytes_per_launch": STAGE_BYTES[name],
                         "achieved_gbs": round(gbs, 1), "frac": round(gbs / peaks()[0], 4)}
    dom = max(stages, key=stages.get)

    # ---- e2e: the Python API with host buffers, copies inside the timed region:
    # the layer stack's c1 step as one graph (DecodeStackGraph), x of every
    # layer from pinned host memory in, every layer's output back
    from nvfp4_gated_deltanet_gb300.graphs import DecodeStackGraph
    xh = torch.empty(n_layers, 1, layers[0].H, dtype=torch.int16).pin_memory()
    xh.copy_(xd[:1].cpu().expand(n_layers, 1, -1))
    oh = torch.empty(n_layers, 1, layers[0].H, dtype=torch.int16).pin_memory()
    sg = DecodeStackGraph(layers, states, 1)
    e2e_steps = max(5, args.steps // 10)
    for it in range(e2e_steps + 2):
        if it == 2:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        out = sg.step(xh)
        oh.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
    e2e_us = (time.perf_counter() - t0) / e2e_steps * 1e6 / n_layers

    extra = {}
    if not args.no_extra:
        for B in (2, 4, 8, 16):
            gB, _ = capture_stack(layers, states, xd, B)
            msB = time_graph(gB, max(10, args.steps // 4), 3)
            usB = msB * 1e3 / n_layers
            extra[f"c{B}"] = {"us_per_layer_step": round(usB, 3),
                              "hbm_gbs": round(step_bytes(B) / (usB * 1e-6) / 1e9, 1),
                              "frac_of_peak": round(step_bytes(B) / (usB * 1e-6) / 1e9 / hbm_peak, 4)}
            del gB
        extra["c1"] = {"us_per_layer_step": round(us_layer, 3), "hbm_gbs": round(gbs_step, 1),
                       "frac_of_peak": round(gbs_step / hbm_peak, 4)}
        # multi-token verify: 4 sequences x 4 candidate tokens, then the commit of all
        extra["verify_b4_r4"] = time_verify(layers, states, xd, 4, 4, max(10, args.steps // 4))
        del layers, states
        torch.cuda.empty_cache()
        # the two-way head-parallel slice (8 key / 16 value heads), benched the same way
        tp = synth.TP2
        n_tp = max(4, -(-4 * l2 // step_bytes(1, tp)) + 1)
        _, tl, ts, tx = make_stack(pkg, synth, n_tp, 16, 16, shape=tp)
        for B in (1, 2, 4, 8, 16):
            gB, _ = capture_stack(tl, ts, tx, B)
            usB = time_graph(gB, max(10, args.steps // 4), 3) * 1e3 / n_tp
            gbsB = step_bytes(B, tp) / (usB * 1e-6) / 1e9
            extra[f"tp2_c{B}"] = {"us_per_layer_step": round(usB, 3), "hbm_gbs": round(gbsB, 1),
                                  "frac_of_peak": round(gbsB / hbm_peak, 4), "layers": n_tp,
                                  "shape": "H2048 Hk8 Hv16 d128 K4 (one rank of two-way head parallelism)"}
            del gB
        del tl, ts
        torch.cuda.empty_cache()
        # BF16-stored recurrent state: same kernels, half the state bytes
        _, bl, bs, bx = make_stack(pkg, synth, n_layers, 16, 16, state_bf16=True)
        for B in (1, 4, 16):
            gB, _ = capture_stack(bl, bs, bx, B)
            usB = time_graph(gB, max(10, args.steps // 4), 3) * 1e3 / n_layers
            gbsB = step_bytes(B, state_bf16=True) / (usB * 1e-6) / 1e9
            extra[f"bf16state_c{B}"] = {"us_per_layer_step": round(usB, 3), "hbm_gbs": round(gbsB, 1),
                                        "frac_of_peak": round(gbsB / hbm_peak, 4)}
            del gB
        del bl, bs
        torch.cuda.empty_cache()
        for B in (64, 128, 256):
            extra[f"batch{B}"] = time_batch(pkg, synth, B, hbm_peak)
            torch.cuda.empty_cache()
        extra["bf16state_batch256"] = time_batch(pkg, synth, 256, hbm_peak, state_bf16=True)
        torch.cuda.empty_cache()
        # KDA-style per-channel recurrent step, 64 heads x 128 (the KDA entry's layer)
        for M in (1, 8, 32):
            for sb in (False, True):
                extra[f"kda_m{M}_{'bf16' if sb else 'f32'}"] = time_kda(pkg, synth, M, 64, 128, sb, hbm_peak, l2,
                                                                        max(10, args.steps // 4))
                torch.cuda.empty_cache()
        for T in (1024, 4096, 16384):
            extra[f"prefill{T}"] = time_prefill(pkg, synth, T)
            torch.cuda.empty_cache()
        for T in (4096, 16384):
            extra[f"prefill{T}_in_proj"] = time_in_proj(pkg, synth, T)
            torch.cuda.empty_cache()

    cpu = None if (args.no_cpu or rank != 0) else cpu_baseline_leg()
    if cpu is not None:
        cpu["all_cores"] = cpu_all_cores_leg()
        cpu["configs"] = cpu_configs_leg()
    line = {
        "metric": METRIC, "value": round(us_layer, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4-w4a4 (fp32 accum) + f32 state", "data": "synthetic",
        "config": headline_config(world),
        "stack": {"layers_per_step": n_layers,
                  "l2_defeat": f"{n_layers} distinct layer instances, {n_layers * per_layer / 1e6:.0f} MB > 4x L2 "
                               f"({l2 / 1e6:.0f} MB)"},
        "hbm_gbs_step": round(gbs_step, 1), "hbm_frac_step": round(gbs_step / hbm_peak, 4),
        "roofline": {"bound": "hbm", "kernel": STAGE_KERNELS[dom], "stage": dom,
                     "achieved": kernels[dom]["achieved_gbs"], "peak": hbm_peak, "unit": "GB/s",
                     "frac": kernels[dom]["frac"], "peak_kind": peak_kind, "traffic": STAGE_TRAFFIC.get(dom),
                     "us_per_launch": kernels[dom]["us_per_launch"], "bytes_per_launch": STAGE_BYTES[dom],
                     "kernels": kernels},
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": int(xh.numel() * 2),
                "d2h_bytes_per_step": int(oh.numel() * 2),
                "path": "DecodeStackGraph (one CUDA graph of every layer's gdn_decode_step through the C ABI), pinned host x in / out back"},
        "gpu_launches": 3 * n_layers * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
