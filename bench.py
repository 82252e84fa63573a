"""Benchmark: one Gemma-3-4B-shaped decode layer of block-quantized matvecs.

A step is one decode layer at batch 1, hidden 2560 (the larql Gemma 3 table's
quantized path): mixed QKV (Q/K Q4_K, V Q6_K) -> O projection (Q4_K
2560x2048) -> FFN gate+up with GELU-tanh (Q4_K 2 x 10240 x 2560) -> FFN down
(Q6_K 2560 x 10240).  Each op feeds the next (q -> O, O's output -> gate+up,
h -> down).  34 layer copies (the model's depth, 2.06 GB of weights) rotate
step by step, so the weights never sit in the 129 MB L2 between uses.

Headline metric: effective weight GB/s = weight-block bytes of the layer per
second (60,518,400 B per step), with us/layer = ms_per_step * 1000.  The
device-timed number replays the decode pass (the layer copies captured in
CUDA graphs, so consecutive launches overlap) with inputs resident; every
graph replayed in the timed region has been replayed before it.

`e2e` times the same C ABI calls with every step's x copied in from pinned
host memory and its layer output copied back to pinned host memory: the
copies on their own streams overlapping the kernels (double-buffered, one
CUDA graph per step), and, as `e2e.direct`, the plain sequence a caller
without graphs issues (copy in, four API calls, copy out, per step), with
the host time spent inside the API calls.

Besides the layer, the default line carries per-launch figures of the
layer's four calls and of the other named workloads (`configs`): a 256 x 2560
Q4_K matvec, the Llama-3-8B FFN in Q4_K and Q8_0 at batch 1, 2, 4, 8, the
262144 x 2560 Q4_K lm_head with its fp16 / fp32 fallbacks, and the Mixtral
MoE FFN; `fusions` compares the fused input norm and activated down input
with the same work unfused.

--impl reference runs the CPU oracle (fp64, all host cores) on the layer:
each step is every row of every matrix of one layer copy; the repo arm's
`cpu_baseline` times the same sample.

--workload selects one of the other named shapes instead of the layer, with
the same JSON line: llama_ffn (SwiGLU FFN 2 x 14336 x 4096 + 4096 x 14336 at
--batch M, --fmt q4k|q80), lm_head (262144 x 2560 Q4_K, batch 1; --softcap C
fuses the final-logit soft-cap C * tanh(y / C) into the store),
mixtral_moe (8 experts, top-2, 16 tokens, Q4_K) and matvec_small (Q4_K 256 x
2560, batch 1).  A step is one call of the workload; weight copies rotate
so that each step reads weights that are not in L2 (at least three times
the L2 size in total, one copy when a single one is larger).

Multi-GPU (torchrun): every rank runs an independent replica (the layer has
no data-path exchange); timing is max over ranks, value is the sum.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

H_, I_, NQ_, NKV_ = 2560, 10240, 2048, 1024
CALL_WEIGHT_BYTES = {"qkv": 6_574_080, "o": 2_949_120, "gateup": 29_491_200, "down": 21_504_000}
# fp32 activations each call reads and writes once (x in, y out)
CALL_ACT_BYTES = {"qkv": 4 * (H_ + NQ_ + 2 * NKV_), "o": 4 * (NQ_ + H_), "gateup": 4 * (H_ + I_),
                  "down": 4 * (I_ + H_)}
LAYER_BYTES = sum(CALL_WEIGHT_BYTES.values())        # 60,518,400
NLAYERS = 34
METRIC = "effective weight GB/s per quantized matvec (decode layer, batch 1)"
WORKLOADS = ("gemma_layer", "llama_ffn", "lm_head", "mixtral_moe", "matvec_small", "prefill_gemm")
CPU_STEPS_MAX = 272                                  # repo arm's oracle sample: layer steps


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8 * NLAYERS)
    ap.add_argument("--warmup", type=int, default=NLAYERS)
    ap.add_argument("--impl", default="lq", choices=["lq", "reference"])
    ap.add_argument("--layers", type=int, default=NLAYERS)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config figures")
    ap.add_argument("--workload", default="gemma_layer", choices=list(WORKLOADS))
    ap.add_argument("--batch", type=int, default=8, help="x rows (llama_ffn, prefill_gemm)")
    ap.add_argument("--fmt", default="q4k", choices=["q4k", "q80"], help="weight format (llama_ffn, prefill_gemm)")
    ap.add_argument("--softcap", type=float, default=0.0,
                    help="final-logit soft-cap fused into the store (lm_head; 0 = none)")
    a = ap.parse_args()
    if a.workload != "gemma_layer":
        if "--steps" not in sys.argv:
            a.steps = 2200 if a.workload == "matvec_small" else 200   # at least two passes over the copies
        if "--warmup" not in sys.argv:
            a.warmup = 20
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    return a


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 and args.impl != "reference":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return ws, rank, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16 tensor throughput in TFLOP/s: the measured bf16 figure (fp16
    runs at the bf16 rate on this part), burst, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 at the same rate)"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            p = [s.strip() for s in l.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx = float(p[1])
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def host_layers(n):
    """n Gemma-3-4B-shaped layers as host arrays (seeded synthetic blocks) and x."""
    import synth
    out = []
    for i in range(n):
        L, x = synth.gemma3_layer(seed=i)
        out.append(L)
        if i == 0:
            x0 = x
    return out, x0


def make_layers(n, dev, host=None):
    """the n layers on the device, gate/up packed (lq_pack_gate_up)."""
    import torch
    import block_quantized_weight_super_gb300 as lq
    import synth
    if host is None:
        host, x0 = host_layers(n)
    else:
        x0 = None
    layers = []
    for L in host:
        d = {k: torch.from_numpy(v).to(dev) for k, v in L.items()}
        rb = lq.lq_row_bytes(lq.LQ_Q4_K, synth.GEMMA3_HIDDEN)
        wgu = torch.empty(2 * synth.GEMMA3_INTER * rb, dtype=torch.uint8, device=dev)
        lq.lq_pack_gate_up(lq.LQ_Q4_K, d["wg"], d["wu"], synth.GEMMA3_INTER, synth.GEMMA3_HIDDEN, wgu)
        d["wgu"] = wgu
        del d["wg"], d["wu"]
        layers.append(d)
    torch.cuda.synchronize()
    return layers, x0


class Layer:
    """buffers and calls of one decode layer through the C ABI."""

    def __init__(self, dev):
        import torch
        f = dict(dtype=torch.float32, device=dev)
        self.x = torch.zeros((1, H_), **f)
        self.q = torch.empty((1, NQ_), **f)
        self.k = torch.empty((1, NKV_), **f)
        self.v = torch.empty((1, NKV_), **f)
        self.o = torch.empty((1, H_), **f)
        self.h = torch.empty((1, I_), **f)
        self.y = torch.empty((1, H_), **f)

    def call(self, name, w, stream, x=None, y=None):
        import block_quantized_weight_super_gb300 as lq
        if name == "qkv":
            lq.lq_qkv_mixed(lq.LQ_Q4_K, w["wq"], NQ_, lq.LQ_Q4_K, w["wk"], NKV_, lq.LQ_Q6_K, w["wv"], NKV_,
                            H_, self.x if x is None else x, self.q, self.k, self.v, 1, stream)
        elif name == "o":
            lq.lq_matvec(lq.LQ_Q4_K, w["wo"], H_, NQ_, self.q, self.o, 1, stream)
        elif name == "gateup":
            lq.lq_ffn_gate_up_act(lq.LQ_Q4_K, w["wgu"], I_, H_, self.o, self.h, 1, lq.LQ_ACT_GEGLU_TANH, stream)
        else:
            lq.lq_matvec(lq.LQ_Q6_K, w["wd"], H_, I_, self.h, self.y if y is None else y, 1, stream)

    def run(self, w, stream, x=None, y=None):
        """the layer's four calls; x / y override the input and output buffers."""
        for name in ("qkv", "o", "gateup", "down"):
            self.call(name, w, stream, x=x, y=y)


def timed_graphs(fn, items, steps, warmup, st):
    """ms per step of fn(item, st) over the rotating items, exactly `steps`
    steps: CUDA graphs of a full pass over the items and of the partial pass
    that completes `steps`; both are replayed (warm) before the timed region,
    the full one for at least `warmup` steps."""
    import torch

    def capture(cs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for w in cs:
                fn(w, st)
        return g

    n = len(items)
    with torch.cuda.stream(st):
        for w in items:               # every launch once outside capture (plans, attributes)
            fn(w, st)
        st.synchronize()
        full = capture(items)
        rem = steps % n
        part = capture(items[:rem]) if rem else None
        for _ in range(max(1, -(-warmup // n))):
            full.replay()
        if part is not None:
            part.replay()
        st.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(steps // n):
            full.replay()
        if part is not None:
            part.replay()
        e1.record(st)
        st.synchronize()
    return e0.elapsed_time(e1) / steps


def bench_lq(args, ws, rank, local, peak):
    import torch
    import block_quantized_weight_super_gb300 as lq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lq.lib()
    hl, x0 = host_layers(args.layers)
    layers, _ = make_layers(args.layers, dev, host=hl)
    st = torch.cuda.Stream(device=dev)
    lay = Layer(dev)
    lay.x.copy_(torch.from_numpy(x0))
    torch.cuda.synchronize()
    rc, bits = lq.lq_device_status()
    assert rc == 0
    n = len(layers)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(local) as clk:
        ms = timed_graphs(lay.run, layers, args.steps, args.warmup, st)
        barrier()
    ms_all = ms
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_all = float(t.item())
    rc, bits = lq.lq_device_status()
    assert rc == 0, "device status after timed region"

    # each of the layer's four launches alone, rotating the layer copies
    # (one graph of n launches), CUDA events on the launching stream
    calls = {}
    for name in ("qkv", "o", "gateup", "down"):
        t = timed_graphs(lambda w, s, nm=name: lay.call(nm, w, s), layers, max(n, args.steps), 3 * n, st)
        nb = CALL_WEIGHT_BYTES[name] + CALL_ACT_BYTES[name]
        calls[name] = {"us": t * 1e3, "alg_bytes": nb, "GB_s": nb / (t * 1e-3) / 1e9,
                       "frac": nb / (t * 1e-3) / 1e9 / peak}

    fusions = None if args.no_configs else fusion_figures(lay, layers, max(n, args.steps), 3 * n, st, dev)
    e2e = None if args.no_e2e else bench_e2e(args, ws, dev, st, lay, layers, x0, barrier)
    return ms_all, calls, fusions, clk.summary(), e2e, hl


def fusion_figures(lay, layers, steps, warmup, st, dev):
    """us per layer copy of the fused input norm and activated down input
    against the same work unfused, on the layer's shapes (rotating copies):
    qkv_rmsnorm: lq_qkv_mixed_rmsnorm vs lq_rmsnorm + lq_qkv_mixed;
    ffn_act: lq_matvec over the packed gate/up rows + lq_matvec_act (the
    activation on down's x-load) vs lq_ffn_gate_up_act + lq_matvec (the
    activation in gate+up's store, the layer's form)."""
    import torch
    import block_quantized_weight_super_gb300 as lq
    import synth
    g = synth.rng(99)
    nw = torch.from_numpy((1.0 + 0.25 * g.standard_normal(H_)).astype(np.float32)).to(dev)
    xn = torch.empty((1, H_), dtype=torch.float32, device=dev)
    gu = torch.empty((1, 2 * I_), dtype=torch.float32, device=dev)
    eps = 1e-6

    def qkv_fused(w, s):
        lq.lq_qkv_mixed_rmsnorm(lq.LQ_Q4_K, w["wq"], NQ_, lq.LQ_Q4_K, w["wk"], NKV_, lq.LQ_Q6_K, w["wv"], NKV_, H_,
                                lay.x, nw, eps, xn, lay.q, lay.k, lay.v, 1, s)

    def qkv_unfused(w, s):
        lq.lq_rmsnorm(lay.x, nw, eps, xn, 1, H_, s)
        lay.call("qkv", w, s, x=xn)

    def ffn_act_down(w, s):
        lq.lq_matvec(lq.LQ_Q4_K, w["wgu"], 2 * I_, H_, lay.o, gu, 1, s)
        lq.lq_matvec_act(lq.LQ_Q6_K, w["wd"], H_, I_, gu, lay.h, lay.y, 1, lq.LQ_ACT_GEGLU_TANH, s)

    def ffn_act_gateup(w, s):
        lay.call("gateup", w, s)
        lay.call("down", w, s)

    out = {}
    for name, fn in (("qkv_rmsnorm_fused", qkv_fused), ("qkv_rmsnorm_unfused", qkv_unfused),
                     ("ffn_act_on_down_load", ffn_act_down), ("ffn_act_in_gate_up", ffn_act_gateup)):
        out[name] = {"us": timed_graphs(fn, layers, steps, warmup, st) * 1e3}
    out["launches"] = {"qkv_rmsnorm_fused": 1, "qkv_rmsnorm_unfused": 2, "ffn_act_on_down_load": 2,
                       "ffn_act_in_gate_up": 2}
    return out


def bench_e2e(args, ws, dev, st, lay, layers, x0, barrier):
    """e2e through the C ABI: every step copies its x in from pinned host
    memory and its layer output back to pinned host memory.

    Graphed: step i's input and output live in device slots i & 1; the copies
    run on their own streams so that they overlap the kernels: step i holds
    [copy-in of step i+1's x] || [layer i] || [copy-out of step i-1's output],
    the copies forked after layer i-1 and joined before layer i+1.  The steps
    of one pass over the layer copies are captured in one CUDA graph (so one
    layer's last kernel and the next one's first keep their programmatic
    dependent launch), and the remainder of K in a second; a copy-in before
    the first step and a copy-out after the last complete the K steps.  Both
    graphs are replayed before the timed region.

    Direct: per step, copy x in, the four API calls, copy the output out, all
    on one stream with no graph (what a caller without graphs pays, host work
    of the calls included)."""
    import torch
    n = len(layers)
    xh = torch.from_numpy(x0).pin_memory()
    yh = torch.empty((1, H_), dtype=torch.float32).pin_memory()
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    xb = [torch.empty_like(lay.x) for _ in range(2)]
    yb = [torch.empty_like(lay.y) for _ in range(2)]
    ng = n if n % 2 == 0 else 2 * n              # a whole number of slot cycles

    def steps_graph(i0, k):                  # steps i0 .. i0+k-1: layer copy i % n, slot i & 1
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(i0, i0 + k):
                c, s = i % n, i & 1
                fork = torch.cuda.Event()
                fork.record(st)
                cin.wait_event(fork)
                cout.wait_event(fork)
                with torch.cuda.stream(cin):
                    xb[s ^ 1].copy_(xh, non_blocking=True)           # the next step's slot
                with torch.cuda.stream(cout):
                    yh.copy_(yb[s ^ 1], non_blocking=True)           # the previous step's slot
                lay.run(layers[c], st, x=xb[s], y=yb[s])
                st.wait_stream(cin)
                st.wait_stream(cout)
        return g

    with torch.cuda.stream(st):
        full = steps_graph(0, ng)
        rem = args.steps % ng
        part = steps_graph(0, rem) if rem else None
        torch.cuda.synchronize()

        def run_steps(k):
            xb[0].copy_(xh, non_blocking=True)
            for _ in range(k // ng):
                full.replay()
            if k % ng:
                part.replay()
            yh.copy_(yb[(k - 1) & 1], non_blocking=True)

        run_steps(max(ng, args.warmup))             # the full graph replayed at least once
        if part is not None:
            run_steps(rem)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        run_steps(args.steps)
        torch.cuda.synchronize()
        t_e2e = (time.perf_counter() - t0) / args.steps

        def direct_steps(k):
            host = 0.0
            for i in range(k):
                lay.x.copy_(xh, non_blocking=True)
                h0 = time.perf_counter()
                lay.run(layers[i % n], st)
                host += time.perf_counter() - h0
                yh.copy_(lay.y, non_blocking=True)
            return host

        direct_steps(max(n, args.warmup))
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        host = direct_steps(args.steps)
        torch.cuda.synchronize()
        t_dir = (time.perf_counter() - t0) / args.steps
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([t_e2e, t_dir], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_e2e, t_dir = float(t[0].item()), float(t[1].item())
    return {"value": ws * LAYER_BYTES / t_e2e / 1e9, "unit": "GB/s", "us_per_layer": t_e2e * 1e6,
            "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(yh.numel() * 4),
            "copies": "own streams, overlapping the kernels (x and output double-buffered); one graph per pass over the layer copies",
            "direct": {"value": ws * LAYER_BYTES / t_dir / 1e9, "unit": "GB/s", "us_per_layer": t_dir * 1e6,
                       "host_us_per_call": host / args.steps / 4 * 1e6,
                       "how": "no graph: per step copy x in, four API calls, copy the output out, one stream"}}


# ---------------------------------------------------------------- the CPU oracle sample

class OracleLayers:
    """the oracle (fp64 C++, all host threads) over the layer copies: a step
    is every row of every matrix of one layer copy (7 matvecs, 60,518,400
    weight bytes), copies taken in turn."""

    def __init__(self, hl):
        import synth
        g = synth.rng(1234)
        self.hl = hl
        self.xs = {"h": synth.activations(g, 1, H_), "q": synth.activations(g, 1, NQ_),
                   "i": synth.activations(g, 1, I_)}
        self.nth = os.cpu_count() or 1

    def step(self, i):
        import oracle
        L = self.hl[i % len(self.hl)]
        xh, xq, xi = self.xs["h"], self.xs["q"], self.xs["i"]
        for fmt, W, cols, x in ((oracle.Q4_K, L["wq"], H_, xh), (oracle.Q4_K, L["wk"], H_, xh),
                                (oracle.Q6_K, L["wv"], H_, xh), (oracle.Q4_K, L["wo"], NQ_, xq),
                                (oracle.Q4_K, L["wg"], H_, xh), (oracle.Q4_K, L["wu"], H_, xh),
                                (oracle.Q6_K, L["wd"], I_, xi)):
            oracle.matvec(fmt, W, W.shape[0], cols, x, self.nth)

    def run(self, steps, warmup):
        for i in range(warmup):
            self.step(i)
        t0 = time.perf_counter()
        for i in range(steps):
            self.step(warmup + i)
        return (time.perf_counter() - t0) / steps

    def describe(self, steps):
        return {"kind": "oracle", "cores": self.nth,
                "sample": f"{steps} layer steps: every row of every matrix of one layer copy per step "
                          f"({LAYER_BYTES} weight bytes), copies in turn, fp64, {self.nth} threads"}


# DRAM bytes (read + write) of one gate+up launch from an ncu capture, valid
# while the sources of that kernel hash to the value they had when it was taken.
GATEUP_TRAFFIC = {"csrc_sha256": "722ebb852addff15d4313d0877a7fde740c31bf4365a4546da611af685a08e73",
                  "bytes": 29_563_392,
                  "source": "profiles/gv_gate_up_q4k_gemma3.md (ncu dram bytes per launch, dram-only capture)"}

# the sources the batch-1 gate+up launch is compiled from
GV_SOURCES = ("lq_codec.cuh", "lq_device.cuh", "lq_group.cuh", "lq_gv.cu", "lq_gv.cuh", "lq_internal.h",
              "lq_qmv.cuh", "lq_stream.cuh")


def csrc_sha256():
    import hashlib
    d = os.path.join(ROOT, "block_quantized_weight_super_gb300", "csrc")
    h = hashlib.sha256()
    for f in GV_SOURCES:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def l2_bytes():
    """L2 size of GPU 0 (129 MB on GB300 when no device is visible)."""
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        pass
    return 129_000_000


def n_copies(nbytes):
    """rotating copies: at least 3x the L2 size in total, one when a single copy is larger."""
    if nbytes > l2_bytes():
        return 1
    return max(1, min(2048, -(-3 * l2_bytes() // max(1, nbytes))))


def clone(d):
    return {k: ([t.clone() for t in v] if isinstance(v, list) else v.clone()) for k, v in d.items()}


# ---------------------------------------------------------------- other workloads

class Workload:
    """one named shape: weight copies, the step (one call of the workload),
    its dominant kernel, and the host-side oracle sample."""

    def __init__(self, args, dev):
        import torch
        import block_quantized_weight_super_gb300 as lq
        import synth
        self.lq, self.dev = lq, dev
        f32 = dict(dtype=torch.float32, device=dev)
        name = args.workload
        self.name = name
        up = lambda a: torch.from_numpy(a).to(dev)
        if name == "llama_ffn":
            fmt = lq.LQ_Q4_K if args.fmt == "q4k" else lq.LQ_Q8_0
            M = args.batch
            W, X = synth.llama_ffn(fmt, M, seed=0)
            H, I = synth.LLAMA_HIDDEN, synth.LLAMA_INTER
            rb = lq.lq_row_bytes(fmt, H)
            wgu = torch.empty(2 * I * rb, dtype=torch.uint8, device=dev)
            lq.lq_pack_gate_up(fmt, up(W["wg"]), up(W["wu"]), I, H, wgu)
            base = {"wgu": wgu, "wd": up(W["wd"])}
            self.bytes = wgu.numel() + base["wd"].numel()
            self.dom_bytes = wgu.numel()
            self.x_host = X
            self.x = up(X)
            self.h = torch.empty((M, I), **f32)
            self.y = torch.empty((M, H), **f32)
            self.desc = (f"Llama-3-8B-shaped SwiGLU FFN, batch {M}, {args.fmt.upper()}: gate+up 2x14336x4096 "
                         f"fused with SwiGLU, down 4096x14336")
            self.dom_name = f"ffn gate+up SwiGLU ({args.fmt.upper()} 2x14336x4096, batch {M})"
            self.launches = 2
            self._gu = lambda w, st: lq.lq_ffn_gate_up_act(fmt, w["wgu"], I, H, self.x, self.h, M, lq.LQ_ACT_SWIGLU, st)
            self._down = lambda w, st: lq.lq_matvec(fmt, w["wd"], H, I, self.h, self.y, M, st)
            self.step = lambda w, st: (self._gu(w, st), self._down(w, st))
            self.dom = self._gu
            self.cpu_jobs = [(fmt, W["wg"], H, X), (fmt, W["wu"], H, X), (fmt, W["wd"], I, np.zeros((M, I), np.float32))]
        elif name == "prefill_gemm":
            fmt = lq.LQ_Q4_K if args.fmt == "q4k" else lq.LQ_Q8_0
            M = args.batch
            W, X = synth.llama_ffn(fmt, M, seed=0)
            H, I = synth.LLAMA_HIDDEN, synth.LLAMA_INTER
            rb = lq.lq_row_bytes(fmt, H)
            wgu = torch.empty(2 * I * rb, dtype=torch.uint8, device=dev)
            lq.lq_pack_gate_up(fmt, up(W["wg"]), up(W["wu"]), I, H, wgu)
            base = {"wgu": wgu, "wd": up(W["wd"])}
            self.bytes = self.dom_bytes = wgu.numel() + base["wd"].numel()
            self.x_host = X
            self.x = up(X)
            self.h = torch.empty((M, I), **f32)
            self.y = torch.empty((M, H), **f32)
            nws = max(lq.lq_gemm_workspace_bytes(M, 2 * I, H), lq.lq_gemm_workspace_bytes(M, H, I))
            self.ws = torch.empty(nws, dtype=torch.uint8, device=dev)
            self.desc = (f"prefill of the Llama-3-8B SwiGLU FFN, {M} x rows, {args.fmt.upper()}: gate+up 2x14336x4096 "
                         f"fused with SwiGLU (lq_gemm_gate_up_act), down 4096x14336 (lq_gemm)")
            self.dom_name = f"prefill FFN ({args.fmt.upper()}, M {M}), gemm_tc_kernel"
            self.dom_flops = 2.0 * M * H * I * 3                   # gate, up, down: useful multiply-adds x 2
            # per call: scale pre-pass, x image, GEMM; the down projection (4096 rows) adds the split-K sum
            self.launches = 7
            self.step = lambda w, st: (lq.lq_gemm_gate_up_act(fmt, w["wgu"], I, H, self.x, self.h, M, lq.LQ_ACT_SWIGLU,
                                                              self.ws, nws, st),
                                       lq.lq_gemm(fmt, w["wd"], H, I, self.h, self.y, M, self.ws, nws, st))
            self.dom = self.step
            self.cpu_jobs = [(fmt, W["wg"], H, X[:1]), (fmt, W["wu"], H, X[:1]),
                             (fmt, W["wd"], I, np.zeros((1, I), np.float32))]
        elif name in ("lm_head", "matvec_small"):
            if name == "lm_head":
                Wn, x = synth.lm_head(0)
                cols = synth.GEMMA3_HIDDEN
                self.desc = "large-vocab lm_head: Q4_K 262144x2560 of an RMS-normed x, batch 1, fp32 logits"
            else:
                Wn, x = synth.matvec_small(0)
                cols = 2560
                self.desc = "single Q4_K matvec 256x2560, batch 1"
            rows = Wn.shape[0]
            base = {"w": up(Wn)}
            self.bytes = self.dom_bytes = Wn.nbytes
            self.x_host = x
            self.x = up(x)
            self.y = torch.empty((1, rows), **f32)
            self.dom_name = f"Q4_K matvec {rows}x{cols}, batch 1"
            self.launches = 1
            cap = args.softcap if name == "lm_head" else 0.0
            if cap > 0:
                self.desc += f", final-logit soft-cap {cap:g} fused into the store"
                self.dom_name += f", soft-cap {cap:g}"
                self.step = lambda w, st: lq.lq_matvec_softcap(lq.LQ_Q4_K, w["w"], rows, cols, self.x, self.y, 1,
                                                               cap, st)
            else:
                self.step = lambda w, st: lq.lq_matvec(lq.LQ_Q4_K, w["w"], rows, cols, self.x, self.y, 1, st)
            self.dom = self.step
            self.cpu_jobs = [(lq.LQ_Q4_K, Wn, cols, x)]
        elif name == "mixtral_moe":
            R, W1, W3, W2, X = synth.mixtral_moe(0)
            E, H = R.shape
            I = W1[0].shape[0]
            T, K = X.shape[0], synth.MIXTRAL_TOPK
            base = {"d1": [up(a) for a in W1], "d3": [up(a) for a in W3], "d2": [up(a) for a in W2]}
            self.R = up(R)
            self.x_host = X
            self.x = up(X)
            self.y = torch.empty((T, H), **f32)
            self.idx = torch.empty((T, K), dtype=torch.int32, device=dev)
            self.wts = torch.empty((T, K), **f32)
            nb = lq.lq_moe_workspace_bytes(E, K, T, H, I)
            self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            self._moe = lambda w, st: lq.lq_moe_ffn(self.R, E, K, lq.LQ_Q4_K, w["d1"], w["d3"], w["d2"], H, I,
                                                     self.x, self.y, T, self.idx, self.wts, self.ws, nb, st)
            self._moe(base, None)
            torch.cuda.synchronize()
            touched = len(set(self.idx.cpu().numpy().ravel().tolist()))
            self.bytes = self.dom_bytes = touched * (W1[0].nbytes + W3[0].nbytes + W2[0].nbytes)
            self.desc = (f"Mixtral-shaped MoE FFN: 8 experts, top-2, hidden 4096, inter 14336, Q4_K, 16 tokens "
                         f"({touched} experts touched; weight bytes count those)")
            self.dom_name = "grouped expert FFN (route + grouped gate+up + grouped down + combine)"
            self.launches = 4
            self.step = self._moe
            self.dom = self._moe
            e0 = int(self.idx[0, 0].item())
            self.cpu_jobs = [(lq.LQ_Q4_K, W1[e0], H, X[:1]), (lq.LQ_Q4_K, W3[e0], H, X[:1]),
                             (lq.LQ_Q4_K, W2[e0], I, np.zeros((1, I), np.float32))]
        else:
            raise ValueError(name)
        ncopy = n_copies(self.bytes)
        self.copies = [base] + [clone(base) for _ in range(ncopy - 1)]
        torch.cuda.synchronize()

    def cpu(self, rows_frac=0.25):
        import oracle
        nth = os.cpu_count() or 1
        nbytes = 0
        t0 = time.perf_counter()
        for fmt, W, cols, xin in self.cpu_jobs:
            r = max(1, int(W.shape[0] * rows_frac))
            oracle.matvec(fmt, W[:r], r, cols, xin, nth)
            nbytes += W[:r].nbytes
        dt = time.perf_counter() - t0
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": nth, "kind": "oracle",
                "sample": f"first {rows_frac * 100:g}% of the rows of the workload's matrices "
                          f"({nbytes} weight bytes), fp64, {nth} threads"}


def bench_workload(args, ws, rank, local, peak, peak_src):
    import torch
    import block_quantized_weight_super_gb300 as lq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lq.lib()
    wl = Workload(args, dev)
    st = torch.cuda.Stream(device=dev)
    rc, _ = lq.lq_device_status()
    assert rc == 0
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed_graphs(wl.step, wl.copies, args.steps, args.warmup, st)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
    ms_all = ms
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_all = float(t.item())
    dom_ms = ms if wl.dom is wl.step else timed_graphs(wl.dom, wl.copies, args.steps, args.warmup, st)
    rc, _ = lq.lq_device_status()
    assert rc == 0, "device status after timed region"
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(np.ascontiguousarray(wl.x_host)).pin_memory()
        yh = torch.empty(tuple(wl.y.shape), dtype=torch.float32).pin_memory()
        n = len(wl.copies)
        with torch.cuda.stream(st):
            for i in range(max(3, min(args.warmup, n))):
                wl.x.copy_(xh, non_blocking=True)
                wl.step(wl.copies[i % n], st)
                yh.copy_(wl.y, non_blocking=True)
            st.synchronize()
            t0 = time.perf_counter()
            for i in range(args.steps):
                wl.x.copy_(xh, non_blocking=True)
                wl.step(wl.copies[i % n], st)
                yh.copy_(wl.y, non_blocking=True)
            st.synchronize()
            t_e2e = (time.perf_counter() - t0) / args.steps
        e2e = {"value": ws * wl.bytes / t_e2e / 1e9, "unit": "GB/s", "us_per_call": t_e2e * 1e6,
               "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(yh.numel() * 4),
               "how": "no graph: per step copy x in, the API call(s), copy the output out, one stream"}
    if rank != 0:
        return
    achieved = wl.dom_bytes / (dom_ms * 1e-3) / 1e9
    line = {"metric": "effective weight GB/s per quantized matvec", "value": ws * wl.bytes / (ms_all * 1e-3) / 1e9,
            "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all,
            "us_per_call": ms_all * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded random blocks)",
            "config": {"workload": wl.desc, "weight_bytes_per_step": wl.bytes, "weight_copies": len(wl.copies),
                       "l2": ("inputs larger than L2" if len(wl.copies) * wl.bytes > l2_bytes() else
                              "inputs NOT larger than L2") +
                             f" ({len(wl.copies)} rotating copies, {len(wl.copies) * wl.bytes / 1e9:.2f} GB)",
                       "parallelism": f"replicas x{ws}"},
            "frac_of_hbm": ws * wl.bytes / (ms_all * 1e-3) / 1e9 / peak,
            "roofline": ({"bound": "hbm", "kernel": wl.dom_name, "achieved": achieved, "peak": peak,
                          "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                          "us_per_launch": dom_ms * 1e3} if not getattr(wl, "dom_flops", None) else
                         {"bound": "tensor", "kernel": wl.dom_name,
                          "achieved": wl.dom_flops / (dom_ms * 1e-3) / 1e12, "peak": tensor_peak()[0],
                          "peak_source": tensor_peak()[1], "unit": "TFLOP/s",
                          "frac": wl.dom_flops / (dom_ms * 1e-3) / 1e12 / tensor_peak()[0], "traffic": None,
                          "alg_flops_per_step": wl.dom_flops, "us_per_launch": dom_ms * 1e3,
                          "note": "useful flops (2 M K N); the kernel runs three fp16 products per useful one"}),
            "clocks": clk.summary(), "e2e": e2e, "gpu_launches": wl.launches * args.steps,
            "cpu_baseline": wl.cpu() if (ws == 1 and not args.no_cpu) else None}
    print(json.dumps(line))


# ---------------------------------------------------------------- per-config figures of the default line

def config_figures(dev, peak):
    """µs per call, GB/s and fraction of HBM for the other named workloads,
    each timed in graphs over rotating weight copies after warm replays."""
    import torch
    import block_quantized_weight_super_gb300 as lq
    import synth
    st = torch.cuda.Stream(device=dev)
    up = lambda a: torch.from_numpy(a).to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = {}

    def fig(ms, nbytes, ncopy):
        return {"us": ms * 1e3, "weight_bytes": nbytes, "GB_s": nbytes / (ms * 1e-3) / 1e9,
                "frac": nbytes / (ms * 1e-3) / 1e9 / peak, "copies": ncopy}

    def steps_for(ncopy):
        return max(40, 2 * ncopy)

    # config 0: Q4_K 256 x 2560, batch 1
    W, x = synth.matvec_small(0)
    base = {"w": up(W)}
    cs = [base] + [clone(base) for _ in range(n_copies(W.nbytes) - 1)]
    xd, yd = up(x), torch.empty((1, 256), **f32)
    ms = timed_graphs(lambda w, s: lq.lq_matvec(lq.LQ_Q4_K, w["w"], 256, 2560, xd, yd, 1, s), cs,
                      steps_for(len(cs)), len(cs), st)
    out["matvec_small_q4k_256x2560_b1"] = fig(ms, W.nbytes, len(cs))
    del cs, base

    # config 2: Llama-3-8B FFN, Q4_K and Q8_0, batch 1, 2, 4, 8 (gate+up SwiGLU then down)
    H, I = synth.LLAMA_HIDDEN, synth.LLAMA_INTER
    for fmt, tag in ((lq.LQ_Q4_K, "q4k"), (lq.LQ_Q8_0, "q80")):
        Wl, X = synth.llama_ffn(fmt, 8, seed=0)
        wgu = torch.empty(2 * I * lq.lq_row_bytes(fmt, H), dtype=torch.uint8, device=dev)
        lq.lq_pack_gate_up(fmt, up(Wl["wg"]), up(Wl["wu"]), I, H, wgu)
        base = {"wgu": wgu, "wd": up(Wl["wd"])}
        nb = wgu.numel() + base["wd"].numel()
        cs = [base] + [clone(base) for _ in range(n_copies(nb) - 1)]
        Xd = up(X)
        for M in (1, 2, 4, 8):
            h, y = torch.empty((M, I), **f32), torch.empty((M, H), **f32)
            xm = Xd[:M]

            def step(w, s, M=M, h=h, y=y, xm=xm):
                lq.lq_ffn_gate_up_act(fmt, w["wgu"], I, H, xm, h, M, lq.LQ_ACT_SWIGLU, s)
                lq.lq_matvec(fmt, w["wd"], H, I, h, y, M, s)
            ms = timed_graphs(step, cs, steps_for(len(cs)), len(cs), st)
            out[f"llama_ffn_{tag}_b{M}"] = fig(ms, nb, len(cs))
        del cs, base, wgu
        torch.cuda.empty_cache()

    # prefill: the Llama-3-8B SwiGLU FFN as GEMMs over M x rows: gate+up
    # (2 x 14336 x 4096, packed pairs) with the activation fused, then down
    # (4096 x 14336); one weight copy each (the x rows re-use it)
    for fmt, tag in ((lq.LQ_Q4_K, "q4k"), (lq.LQ_Q8_0, "q80")):
        Wl, _ = synth.llama_ffn(fmt, 1, seed=1)
        wgu = torch.empty(2 * I * lq.lq_row_bytes(fmt, H), dtype=torch.uint8, device=dev)
        lq.lq_pack_gate_up(fmt, up(Wl["wg"]), up(Wl["wu"]), I, H, wgu)
        wd = up(Wl["wd"])
        nbw = wgu.numel() + wd.numel()
        for M in (64, 128, 512):
            Xg = torch.randn((M, H), generator=torch.Generator(device=dev).manual_seed(M), device=dev)
            Hh, Yd = torch.empty((M, I), **f32), torch.empty((M, H), **f32)
            nws = max(lq.lq_gemm_workspace_bytes(M, 2 * I, H), lq.lq_gemm_workspace_bytes(M, H, I))
            wsp = torch.empty(nws, dtype=torch.uint8, device=dev)

            def step(w, s, M=M, Xg=Xg, Hh=Hh, Yd=Yd, wsp=wsp, nws=nws):
                lq.lq_gemm_gate_up_act(fmt, wgu, I, H, Xg, Hh, M, lq.LQ_ACT_SWIGLU, wsp, nws, s)
                lq.lq_gemm(fmt, wd, H, I, Hh, Yd, M, wsp, nws, s)
            ms = timed_graphs(step, [None], 20, 3, st)
            out[f"prefill_ffn_{tag}_M{M}"] = dict(fig(ms, nbw, 1), tflops=6.0 * M * H * I / (ms * 1e-3) / 1e12,
                                                   what="gate+up 2x14336x4096 with SwiGLU (lq_gemm_gate_up_act) "
                                                        "+ down 4096x14336 (lq_gemm)")
            if M == 512 and tag == "q4k":
                def step_mv(w, s, M=M, Xg=Xg, Hh=Hh, Yd=Yd):
                    lq.lq_ffn_gate_up_act(fmt, wgu, I, H, Xg, Hh, M, lq.LQ_ACT_SWIGLU, s)
                    lq.lq_matvec(fmt, wd, H, I, Hh, Yd, M, s)
                ms = timed_graphs(step_mv, [None], 10, 3, st)
                out[f"prefill_ffn_batched_{tag}_M{M}"] = dict(fig(ms, nbw, 1), tflops=6.0 * M * H * I / (ms * 1e-3) / 1e12,
                                                               what="the same through lq_ffn_gate_up_act + lq_matvec "
                                                                    "(8 x rows per pass)")
            del Xg, Hh, Yd, wsp
        del wgu, wd
        torch.cuda.empty_cache()

    # config 3: lm_head Q4_K 262144 x 2560, batch 1 (one copy: larger than L2)
    W, x = synth.lm_head(0)
    wd, xd = up(W), up(x)
    yd = torch.empty((1, W.shape[0]), **f32)
    ms = timed_graphs(lambda w, s: lq.lq_matvec(lq.LQ_Q4_K, w, W.shape[0], 2560, xd, yd, 1, s), [wd], 40, 5, st)
    out["lm_head_q4k_262144x2560_b1"] = fig(ms, W.nbytes, 1)
    del wd
    torch.cuda.empty_cache()
    # the non-quantized lm_head fallbacks of the same shape (fp16, fp32 weights;
    # seeded device-side draws: the values do not change the time)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    for dt, name, f in ((torch.float16, "f16", lq.lq_gemv_f16), (torch.float32, "f32", lq.lq_gemv_f32)):
        Wt = (0.05 * torch.randn((W.shape[0], 2560), generator=gen, device=dev, dtype=torch.float32)).to(dt)
        ms = timed_graphs(lambda w, s, f=f: f(w, w.shape[0], 2560, xd, yd, 1, s), [Wt], 40, 5, st)
        out[f"lm_head_{name}_262144x2560_b1"] = fig(ms, Wt.numel() * Wt.element_size(), 1)
        del Wt
        torch.cuda.empty_cache()

    # config 4: Mixtral MoE FFN, 8 experts, top-2, 16 tokens, Q4_K
    R, W1, W3, W2, X = synth.mixtral_moe(0)
    E, Hm = R.shape
    Im = W1[0].shape[0]
    T, K = X.shape[0], synth.MIXTRAL_TOPK
    w = {"d1": [up(a) for a in W1], "d3": [up(a) for a in W3], "d2": [up(a) for a in W2]}
    Rd, Xd = up(R), up(X)
    Y = torch.empty((T, Hm), **f32)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    wts = torch.empty((T, K), **f32)
    nbw = lq.lq_moe_workspace_bytes(E, K, T, Hm, Im)
    wsp = torch.empty(nbw, dtype=torch.uint8, device=dev)
    moe = lambda ww, s: lq.lq_moe_ffn(Rd, E, K, lq.LQ_Q4_K, ww["d1"], ww["d3"], ww["d2"], Hm, Im, Xd, Y, T,
                                      idx, wts, wsp, nbw, s)
    moe(w, None)
    torch.cuda.synchronize()
    touched = len(set(idx.cpu().numpy().ravel().tolist()))
    ms = timed_graphs(moe, [w], 40, 5, st)
    out["mixtral_moe_q4k_8x14336x4096_top2_t16"] = dict(
        fig(ms, touched * (W1[0].nbytes + W3[0].nbytes + W2[0].nbytes), 1), experts_touched=touched)
    del w
    torch.cuda.empty_cache()
    rc, _ = lq.lq_device_status()
    assert rc == 0, "device status after the config figures"
    return out


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    peak, peak_src = peaks()
    base = {"metric": METRIC, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded random Q4_K/Q6_K blocks)",
            "config": {"workload": "Gemma-3-4B-shaped decode layer, batch 1, hidden 2560: QKV "
                                   "(Q/K Q4_K, V Q6_K), O Q4_K, gate+up Q4_K GEGLU-tanh, down Q6_K",
                       "layer_weight_bytes": LAYER_BYTES, "layer_copies": args.layers,
                       "l2": ("inputs larger than L2" if args.layers * LAYER_BYTES > l2_bytes() else
                              "inputs NOT larger than L2") +
                             f" ({args.layers} rotating layer copies, {args.layers * LAYER_BYTES / 1e9:.2f} GB)",
                       "parallelism": f"replicas x{ws}"}}
    if args.workload != "gemma_layer":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the default workload"}))
            return
        bench_workload(args, ws, rank, local, peak, peak_src)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        hl, _ = host_layers(args.layers)
        ol = OracleLayers(hl)
        dt = ol.run(args.steps, args.warmup)
        v = LAYER_BYTES / dt / 1e9
        cb = dict(ol.describe(args.steps), value=v, unit="GB/s")
        line = dict(base, impl="reference", value=v, ms_per_step=dt * 1e3, n_gpus=1,
                    cpu_baseline=cb, e2e={"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0})
        print(json.dumps(line))
        return

    ms, calls, fusions, clocks, e2e, hl = bench_lq(args, ws, rank, local, peak)
    import torch
    configs = None if (args.no_configs or ws > 1) else config_figures(torch.device("cuda", local), peak)
    if rank != 0:
        return
    value = ws * LAYER_BYTES / (ms * 1e-3) / 1e9
    g = calls["gateup"]
    cb = None
    if ws == 1 and not args.no_cpu:
        ol = OracleLayers(hl)
        k = min(args.steps, CPU_STEPS_MAX)
        dt = ol.run(k, 1)
        cb = dict(ol.describe(k), value=LAYER_BYTES / dt / 1e9, unit="GB/s")
    traffic = GATEUP_TRAFFIC["bytes"] if GATEUP_TRAFFIC["csrc_sha256"] == csrc_sha256() else None
    line = dict(base, value=value, ms_per_step=ms, us_per_layer=ms * 1e3,
                frac_of_hbm=value / peak,
                roofline={"bound": "hbm", "kernel": "ffn gate+up GEGLU (Q4_K 2x10240x2560), gv_kernel<1>",
                          "achieved": g["GB_s"], "peak": peak, "peak_source": peak_src,
                          "unit": "GB/s", "frac": g["frac"], "traffic": traffic,
                          "traffic_source": GATEUP_TRAFFIC["source"],
                          "alg_bytes_per_launch": g["alg_bytes"], "us_per_launch": g["us"]},
                layer_calls=calls, fusions=fusions, configs=configs,
                clocks=clocks, e2e=e2e, gpu_launches=4 * args.steps, cpu_baseline=cb)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
