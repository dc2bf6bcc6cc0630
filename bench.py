#!/usr/bin/env python
"""Throughput of the Qwen3-0.6B-shape forward hot path on GB300.

Workload (one "step"): the 28-layer Qwen3-0.6B shape (vocab 151936, hidden
1024, 16 q / 8 kv heads of 128, intermediate 3072) in bf16 with the two-shard
tensor-parallel layout, random-init N(0, 0.02) weights, prefill of 8 sequences
x 2048 tokens (ids uniform over the vocab), then 128 greedy decode steps for
the 8 sequences writing the KV cache.  Every step runs the whole path:
embedding, 28 decoder layers (add+RMSNorm, QKV GEMM, QK-norm + RoPE + KV
store, attention, o_proj, add+RMSNorm, gate_up + SiluAndMul, down), final
norm, lm_head on the last token of each sequence, greedy argmax.

value = tokens processed (16384 prefill + 1024 decoded) per second, timed with
CUDA events over exactly --steps steps after --warmup steps.  The prefill and
decode phases are each captured once in a CUDA graph; the decode graph holds
all 128 steps (each step feeds its argmax to the next on the device).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs its own replica of the workload (the
sequences are independent; no collective on the data path) and value sums
the ranks' tokens over the slowest rank's time.  --impl reference times the
CPU oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "Qwen3-0.6B-shape tokens/s (decode, prefill) on 1 GB300; % HBM / tensor roofline"
UNIT = "tokens/s"
WORKLOAD = "model_prefill_decode"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-layers", type=int, default=4)
    ap.add_argument("--cpu-sample-tokens", type=int, default=2048)
    ap.add_argument("--profile-window", action="store_true",
                    help="after the timed region, run one more step between cudaProfilerStart/Stop "
                         "(for ncu --profile-from-start off)")
    ap.add_argument("--profile-kernel", choices=["decode.attention", "prefill.gemm_gate_up_silu"], default=None,
                    help="launch only this kernel, --profile-reps times, on inputs of the workload's shape "
                         "(random values, mean decode context) and exit: a small case for ncu section captures")
    ap.add_argument("--profile-reps", type=int, default=3)
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: timing barrier and max over ranks)
# ----------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# per-kernel timing probe (CUDA events recorded on the launching stream)
# ----------------------------------------------------------------------------

class KernelProbe:
    """Records timing events around selected launches (inside CUDA graphs when
    the events are external, i.e. captured as event-record nodes)."""

    def __init__(self, layers, external: bool):
        self.layers = set(layers)
        self.external = external
        self.enabled = True
        self.records = {}

    def __call__(self, name, layer):
        if not self.enabled or (layer >= 0 and layer not in self.layers):
            return contextlib.nullcontext()
        return self._rec(name)

    @contextlib.contextmanager
    def _rec(self, name):
        kw = {"enable_timing": True}
        if self.external:
            kw["external"] = True
        e0, e1 = torch.cuda.Event(**kw), torch.cuda.Event(**kw)
        e0.record()
        yield
        e1.record()
        self.records.setdefault(name, []).append((e0, e1))

    def mean_ms(self):
        return {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in self.records.items()}


def external_events_supported() -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


# ----------------------------------------------------------------------------
# the workload on the GPU
# ----------------------------------------------------------------------------

class Workload:
    def __init__(self, device="cuda"):
        import seeded_inputs as si
        from qwen3_transformer_forward_gb300 import build as B
        from qwen3_transformer_forward_gb300 import model as M
        B.build()
        self.si, self.M = si, M
        w = si.workload(WORKLOAD)
        self.w = w
        self.m = m = w.model
        self.seq_lens = list(w.seq_lens)
        self.S = w.decode_steps
        self.B = len(self.seq_lens)
        self.params = M.load_params(m, device=device)
        self.b = si.prefill_batch(m, self.seq_lens, extra_capacity=self.S)
        self.max_context = max(self.seq_lens) + self.S
        self.fwd = M.Qwen3Forward(m, self.params, max_tokens=sum(self.seq_lens), num_slots=self.b.num_slots,
                                  max_seqs=self.B, max_context=self.max_context, device=device)
        self.pctx = M.to_device_prefill(self.b, device)
        cap = self.b.capacity
        base = torch.tensor([sum(cap[:i]) for i in range(self.B)], dtype=torch.int64)
        steps = torch.arange(self.S, dtype=torch.int64)[:, None]
        L0 = torch.tensor(self.seq_lens, dtype=torch.int64)[None, :]
        pos = L0 + steps
        self.host_decode = {"positions": pos, "context_lens": (pos + 1).to(torch.int32),
                            "slots": base[None, :] + pos}
        self.dpos = pos.to(device)
        self.dcl = self.host_decode["context_lens"].to(device)
        self.dslots = self.host_decode["slots"].to(device)
        self.dbase = base.to(torch.int32).to(device)
        self.gen = torch.zeros(self.S + 1, self.B, dtype=torch.int64, device=device)
        self.g_prefill = None
        self.g_decode = None

    # one phase each
    def prefill_phase(self):
        _, nt = self.fwd.prefill(self.pctx)
        self.gen[0].copy_(nt)

    def decode_phase(self, probe_steps=()):
        M, fwd = self.M, self.fwd
        for s in range(self.S):
            if fwd.probe is not None:
                fwd.probe.enabled = s in probe_steps
            ctx = M.DecodeContext(fwd.next_tokens[:self.B], self.dpos[s], self.dcl[s], self.dslots[s], self.dbase,
                                  self.max_context)
            fwd.decode(ctx)
            self.gen[s + 1].copy_(fwd.next_tokens[:self.B])
        if fwd.probe is not None:
            fwd.probe.enabled = True

    def capture(self, probe=None, probe_steps=()):
        """Eager warm-up, then one CUDA graph per phase."""
        self.fwd.probe = None
        self.prefill_phase()
        self.decode_phase()
        torch.cuda.synchronize()
        self.fwd.probe = probe
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        self.g_prefill = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_prefill, stream=s):
            self.prefill_phase()
        self.g_decode = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_decode, stream=s):
            self.decode_phase(probe_steps)
        self.fwd.probe = None
        torch.cuda.synchronize()

    def step(self, mid_event=None):
        self.g_prefill.replay()
        if mid_event is not None:
            mid_event.record()
        self.g_decode.replay()

    # algorithmic work per launch of each probed kind: (bound, amount, unit)
    def work(self):
        m = self.m
        T = sum(self.seq_lens)
        H, I, hd, nh, nkv, V = m.hidden, m.intermediate, m.head_dim, m.n_heads, m.n_kv_heads, m.vocab
        qkvw = (nh + 2 * nkv) * hd
        causal_pairs = sum(L * (L + 1) // 2 for L in self.seq_lens)
        B = self.B
        mean_ctx = statistics.mean(L + s + 1 for s in range(self.S) for L in self.seq_lens)
        gemm_b = lambda M_, N_, K_: 2.0 * (N_ * K_ + M_ * K_ + M_ * N_)  # noqa: E731
        return {
            "prefill.gemm_qkv": ("tensor", 2.0 * T * qkvw * H),
            "prefill.gemm_o": ("tensor", 2.0 * T * H * nh * hd),
            "prefill.gemm_gate_up_silu": ("tensor", 2.0 * T * 2 * I * H),
            "prefill.gemm_down": ("tensor", 2.0 * T * H * I),
            "prefill.attention": ("tensor", 4.0 * hd * nh * causal_pairs),
            "prefill.add_rmsnorm": ("hbm", 2.0 * T * H * 4),
            "prefill.qkv_norm_rope_store_kv": ("hbm", 2.0 * T * (qkvw + nh * hd + 2 * nkv * hd) + 16.0 * T),
            "decode.gemm_qkv": ("hbm", gemm_b(B, qkvw, H)),
            "decode.add_rmsnorm_gemm_qkv": ("hbm", gemm_b(B, qkvw, H) + 2.0 * 3 * B * H),
            "decode.add_rmsnorm_gemm_gate_up": ("hbm", 2.0 * (2 * I * H + B * H + B * I) + 2.0 * 3 * B * H),
            "decode.gemm_o": ("hbm", gemm_b(B, H, nh * hd)),
            "decode.gemm_gate_up_silu": ("hbm", 2.0 * (2 * I * H + B * H + B * I)),
            "decode.gemm_down": ("hbm", gemm_b(B, H, I)),
            # with the QK-norm + RoPE + KV store folded in: the QKV rows in, the new k/v rows out
            "decode.attention": ("hbm", 2.0 * 2 * nkv * hd * B * mean_ctx + 2.0 * B * nh * hd
                                 + 2.0 * B * qkvw + 2.0 * 2 * B * nkv * hd + 16.0 * B),
            "decode.add_rmsnorm": ("hbm", 2.0 * B * H * 4),
            "decode.qkv_norm_rope_store_kv": ("hbm", 2.0 * B * (qkvw + nh * hd + 2 * nkv * hd) + 16.0 * B),
            # one persistent kernel per decode step: every layer's weights, the K/V
            # rows each sequence attends to, the new K/V rows, the activations
            "decode.layers": ("hbm", m.n_layers * (2.0 * (qkvw * H + H * nh * hd + 2 * I * H + H * I)
                                                   + 2.0 * 2 * nkv * hd * B * mean_ctx + 2.0 * 2 * nkv * hd * B
                                                   + 2.0 * B * (4 * H + qkvw + nh * hd + I))),
            "lm_head": ("hbm", 2.0 * V * H + 2.0 * B * V),
            "embed_vocab": ("hbm", 2.0 * 2 * T * H + 8.0 * T),
        }

    def launches_per_step(self, kind):
        nl = self.m.n_layers
        fused_norm = self.fwd.norm_fusion_ok(self.B)
        per_layer = {"add_rmsnorm": 0 if fused_norm and kind.startswith("decode.") else 2}
        base = kind.split(".", 1)[-1]
        if kind in ("lm_head", "embed_vocab"):
            return 1 + self.S
        if kind == "decode.layers":
            return self.S
        n = per_layer.get(base, 1) * nl
        return n * (self.S if kind.startswith("decode.") else 1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "tensor": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "tensor_burst": p["bf16_tflops"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "tensor": 1700.0, "tensor_burst": 1900.0, "source": "fallback"}


def attention_traffic_from_profile():
    """dram bytes per launch of the decode attention kernel from its committed ncu
    summary, or None when attention.cu changed since that capture."""
    import hashlib
    import re
    prof = os.path.join(ROOT, "profiles", "decode_attention_bench_shape.md")
    src = os.path.join(ROOT, "qwen3_transformer_forward_gb300", "csrc", "attention.cu")
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        text = f.read()
    with open(src, "rb") as f:
        src_sha1 = hashlib.sha1(f.read()).hexdigest()
    m_b = re.search(r"dram_bytes_per_launch = (\d+)", text)
    m_h = re.search(r"attention\.cu sha1 = ([0-9a-f]{40})", text)
    if not m_b or not m_h or src_sha1 != m_h.group(1):
        return None
    return int(m_b.group(1))


def attention_roofline(wl, peaks, reps=5):
    """Decode attention alone: one CUDA graph of 28 back-to-back launches, one per
    layer's KV cache (2 GB together, larger than L2), on the decode step halfway
    through the run.  Duration = graph time / launches (events on the replay stream)."""
    from qwen3_transformer_forward_gb300 import _lib as L
    fwd, m = wl.fwd, wl.m
    s = wl.S // 2
    B = wl.B
    cl, base = wl.dcl[s], wl.dbase
    out = fwd.attn[:B]

    qkv, pos, slots = fwd.qkv[:B], wl.dpos[s], wl.dslots[s]

    def chain():   # (stores k/v rows from the qkv buffer, the last decode step's, at step s's slots; the next replay of the step rewrites them)
        for l in range(m.n_layers):
            p = wl.params.layers[l]
            L.attention_decode_rope(qkv, m.n_heads, m.n_kv_heads, m.head_dim, m.tp, pos, fwd.cos_sin, p.q_norm,
                                    p.k_norm, m.eps, slots, fwd.k_cache[l], fwd.v_cache[l], fwd.err, cl, base,
                                    wl.max_context, fwd.scale, out, fwd.workspace, history_ready=True)

    chain()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        chain()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    L.device_error()
    us = e0.elapsed_time(e1) * 1e3 / (reps * m.n_layers)
    ctx = [L0 + s + 1 for L0 in wl.seq_lens]
    hd, nh, nkv = m.head_dim, m.n_heads, m.n_kv_heads
    qkvw = (nh + 2 * nkv) * hd
    algo = 2.0 * 2 * nkv * hd * sum(ctx) + 2.0 * B * nh * hd + 2.0 * B * qkvw + 2.0 * 2 * B * nkv * hd + 16.0 * B
    achieved = algo / (us * 1e-6) / 1e9
    traffic = attention_traffic_from_profile()
    if traffic is not None:   # the capture ran at the mean context: scale to this one
        traffic = round(traffic * sum(ctx) / (B * (statistics.mean(wl.seq_lens) + wl.S // 2)))
    return {"kernel": "decode.attention", "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 3), "traffic": traffic,
            "algorithmic_bytes": round(algo), "us_per_launch": round(us, 2),
            "peak_source": f"{peaks['source']} (HBM copy)",
            "timing": f"{m.n_layers} back-to-back launches over the {m.n_layers} layers' KV caches (larger than L2), "
                      f"decode step {s}, one CUDA graph replayed {reps} times, events on the replay stream"}


def run_ours(args, rank, world, local):
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    from qwen3_transformer_forward_gb300 import _lib as L
    wl = Workload(device)
    ext = external_events_supported()
    probe = KernelProbe(layers=(3, 17), external=True) if ext else None
    probe_steps = (0, 42, 85, 127)
    wl.capture(probe=probe, probe_steps=probe_steps)
    L.device_error()
    tokens_per_step = sum(wl.seq_lens) + wl.S * wl.B

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    barrier(world)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    e0.record()
    starts = []
    for i in range(args.steps):
        st = torch.cuda.Event(enable_timing=True)
        st.record()
        starts.append(st)
        wl.step(mids[i])
        ends[i].record()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    L.device_error()
    ms_total = e0.elapsed_time(e1)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    prefill_ms = statistics.mean(starts[i].elapsed_time(mids[i]) for i in range(args.steps))
    decode_ms = statistics.mean(mids[i].elapsed_time(ends[i]) for i in range(args.steps))
    value = tokens_per_step * world / (ms_total / 1e3 / args.steps)

    peaks = load_peaks()
    kernels = {}
    roofline = None
    probe_method = "event-record nodes inside the timed graphs (last timed step)"
    if probe is None:
        # this torch cannot capture timing events into a graph: time the same
        # launches in one eager step right after the timed region instead
        probe = KernelProbe(layers=(3, 17), external=False)
        wl.fwd.probe = probe
        wl.prefill_phase()
        wl.decode_phase(probe_steps)
        wl.fwd.probe = None
        torch.cuda.synchronize()
        probe_method = "CUDA events around the launches of one eager step after the timed region"
    if probe is not None:
        work = wl.work()
        means = probe.mean_ms()
        for name, ms in means.items():
            if name not in work:
                continue
            bound, amount = work[name]
            total = ms * wl.launches_per_step(name)
            if bound == "hbm":
                achieved = amount / (ms / 1e3) / 1e9
                peak, unit = peaks["hbm"], "GB/s"
            else:
                achieved = amount / (ms / 1e3) / 1e12
                peak, unit = peaks["tensor"], "TFLOP/s"
            kernels[name] = {"bound": bound, "us_per_launch": round(ms * 1e3, 2), "launches_per_step":
                             wl.launches_per_step(name), "ms_per_step": round(total, 3), "achieved": round(achieved, 1),
                             "peak": peak, "unit": unit, "frac": round(achieved / peak, 3)}
        if kernels:
            dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
            kd = kernels[dom]
            roofline = {"kernel": dom, "bound": kd["bound"], "achieved": kd["achieved"], "peak": kd["peak"],
                        "unit": kd["unit"], "frac": kd["frac"], "traffic": None,
                        "peak_source": f"{peaks['source']} ({'HBM copy' if kd['bound'] == 'hbm' else 'bf16 sustained'})",
                        "timing": probe_method}
            if dom == "decode.attention":
                roofline = attention_roofline(wl, peaks)

    if args.profile_window:
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        wl.step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(wl, args, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded), random-init weights",
        "config": {"workload": "qwen3-0.6b-shape 28 layers, tp=2 layout, prefill 8x2048 + 128 greedy decode steps x 8",
                   "tokens_per_step": tokens_per_step, "prefill_tokens": sum(wl.seq_lens),
                   "decode_tokens": wl.S * wl.B, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1.19 GB weights and 2 GB KV cache streamed every step)",
                   "graphs": "prefill and the 128-step decode loop each one CUDA graph"},
        "prefill_tok_s": round(sum(wl.seq_lens) / (prefill_ms / 1e3), 1),
        "decode_tok_s": round(wl.S * wl.B / (decode_ms / 1e3), 1),
        "prefill_ms": round(prefill_ms, 3), "decode_ms": round(decode_ms, 3),
        "roofline": roofline, "kernels": kernels, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
        "gpu_launches": count_launches(wl),
    }
    return out


def count_launches(wl):
    """Kernels of ours launched per step (counted from the call sequence)."""
    from qwen3_transformer_forward_gb300 import _lib as L
    m = wl.m
    per_layer = 2 + 1 + 1 + 1 + 1 + 1 + 1   # 2 norms, qkv gemm, rope/kv, attention, o, gate_up, down
    # decode with few tokens: both norms run inside the GEMVs they feed; in bf16 the
    # QK-norm + RoPE + KV store runs inside decode attention
    dec_layer = per_layer - 2 if wl.fwd.norm_fusion_ok(wl.B) else per_layer
    if wl.fwd.dtype == torch.bfloat16 and m.head_dim == 128:
        dec_layer -= 1
    # split-K sums and the split-KV merge happen inside the GEMM and attention kernels
    prefill = 1 + m.n_layers * per_layer + 1 + 3     # embed, layers, final norm, gather + gemm + argmax
    lm_dec = 2                                       # gemm + argmax
    if wl.fwd.fused_decode_ok(wl.B):
        decode = 1 + 1 + lm_dec                      # embed, all layers in one kernel, lm_head
    else:
        decode = 1 + m.n_layers * dec_layer + 1 + lm_dec
    return prefill + wl.S * decode


def run_e2e(wl, args, world):
    """Same step through the public API with host inputs: H2D copies of the
    step's inputs from pinned memory and a D2H read of the generated tokens
    inside the timed region."""
    b = wl.b
    host = {"ids": b.ids, "positions": b.positions, "cu_seqlens": b.cu_seqlens, "slot_mapping": b.slot_mapping,
            "seq_base": b.seq_base, "last_idx": b.last_idx}
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dec_host = {"positions": wl.host_decode["positions"].pin_memory(),
                "context_lens": wl.host_decode["context_lens"].pin_memory(),
                "slots": wl.host_decode["slots"].pin_memory()}
    dev = {"ids": wl.pctx.ids, "positions": wl.pctx.positions, "cu_seqlens": wl.pctx.cu_seqlens,
           "slot_mapping": wl.pctx.slot_mapping, "seq_base": wl.pctx.seq_base, "last_idx": wl.pctx.last_idx}
    out_host = torch.empty_like(wl.gen, device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values()) + \
        sum(v.numel() * v.element_size() for v in dec_host.values())
    d2h = out_host.numel() * out_host.element_size()

    def one():
        for k in pinned:
            dev[k].copy_(pinned[k], non_blocking=True)
        wl.dpos.copy_(dec_host["positions"], non_blocking=True)
        wl.dcl.copy_(dec_host["context_lens"], non_blocking=True)
        wl.dslots.copy_(dec_host["slots"], non_blocking=True)
        wl.step()
        out_host.copy_(wl.gen, non_blocking=True)

    one()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(args.steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    tokens = (sum(wl.seq_lens) + wl.S * wl.B) * world * args.steps
    return {"value": round(tokens / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "wall_s": round(wall, 3)}


# ----------------------------------------------------------------------------
# the CPU oracle on a bounded sample of the same workload
# ----------------------------------------------------------------------------

def cpu_sample_setup(n_layers_sample: int):
    import oracle as O
    import seeded_inputs as si
    w = si.workload(WORKLOAD)
    m = w.model
    weights = O.load_weights(m, layers=n_layers_sample)
    cos_sin = O.rope_cos_sin(m.max_position, m.head_dim, m.rope_theta)
    return m, weights, cos_sin


def cpu_sample_run(m, weights, cos_sin, n_tokens: int):
    """Prefill of one sequence of n_tokens through the sampled layers, final norm,
    lm_head of the last token; returns (seconds for the 28-layer model, detail)."""
    import numpy as np
    import oracle as O
    import seeded_inputs as si
    nl = len(weights.layers)
    b = si.prefill_batch(m, [n_tokens])
    cache = O.KVCache(nl, b.num_slots, m.n_kv_heads, m.head_dim, m.tp)
    ctx = O.AttnContext(True, b.slot_mapping.numpy(), cu_seqlens=b.cu_seqlens.numpy())
    t0 = time.perf_counter()
    h = O.vocab_parallel_embedding(b.ids.numpy(), weights.embed, m.tp)
    t1 = time.perf_counter()
    res = None
    for l in range(nl):
        h, res = O.decoder_layer(m, weights.layers[l], l, b.positions.numpy(), h, res, ctx, cache, *cos_sin)
    t2 = time.perf_counter()
    h, _ = O.add_rms_norm(h, res, weights.final_norm, m.eps, m.dtype)
    lg = O.compute_logits(m, weights.embed, h, m.tp, b.cu_seqlens.numpy())
    O.greedy(lg)
    t3 = time.perf_counter()
    model_s = (t1 - t0) + (t2 - t1) * m.n_layers / nl + (t3 - t2)
    return model_s, t3 - t0


def cpu_baseline(args):
    m, weights, cos_sin = cpu_sample_setup(args.cpu_sample_layers)
    model_s, wall = cpu_sample_run(m, weights, cos_sin, args.cpu_sample_tokens)
    n = args.cpu_sample_tokens
    return {"value": round(n / model_s, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"prefill of 1 sequence x {n} tokens through {args.cpu_sample_layers} of the 28 layers, "
                      f"embedding, final norm, lm_head of the last token; layer time scaled x "
                      f"{m.n_layers}/{args.cpu_sample_layers} to the full model ({wall:.1f} s of CPU work, "
                      f"numpy float64, threads = all host cores)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    m, weights, cos_sin = cpu_sample_setup(args.cpu_sample_layers)
    n = args.cpu_sample_tokens
    for _ in range(args.warmup):
        cpu_sample_run(m, weights, cos_sin, n)
    times = []
    walls = []
    for _ in range(args.steps):
        s, w = cpu_sample_run(m, weights, cos_sin, n)
        times.append(s)
        walls.append(w)
    ms_step = statistics.mean(times) * 1e3
    value = n / (ms_step / 1e3)
    sample = (f"each step: prefill of 1 sequence x {n} tokens through {args.cpu_sample_layers} of the 28 layers, "
              f"embedding, final norm, lm_head of the last token; layer time scaled x "
              f"{m.n_layers}/{args.cpu_sample_layers}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded), random-init weights",
            "config": {"workload": "qwen3-0.6b-shape 28 layers, tp=2 layout, prefill 8x2048 + 128 greedy decode "
                                   "steps x 8 (bounded CPU sample, see cpu_baseline.sample)"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_kernel(args):
    """One kernel of the workload on inputs of its shape, for a small ncu capture."""
    import seeded_inputs as si
    from qwen3_transformer_forward_gb300 import build as B
    from qwen3_transformer_forward_gb300 import _lib as L
    B.build()
    w = si.workload(WORKLOAD)
    m = w.model
    seqs, S = list(w.seq_lens), w.decode_steps
    nb, nh, nkv, hd = len(seqs), m.n_heads, m.n_kv_heads, m.head_dim
    cap = max(seqs) + S
    g = torch.Generator(device="cuda").manual_seed(0)
    rnd = lambda *shape: torch.randn(*shape, device="cuda", generator=g).to(torch.bfloat16)  # noqa: E731
    if args.profile_kernel == "decode.attention":   # with the folded QK-norm + RoPE + KV store
        kc, vc = rnd(nb * cap, nkv, hd), rnd(nb * cap, nkv, hd)
        qkv = rnd(nb, (nh + 2 * nkv) * hd)
        gamma = torch.ones(hd, dtype=torch.bfloat16, device="cuda")
        ctx = torch.tensor([L0 + S // 2 for L0 in seqs], dtype=torch.int32, device="cuda")
        base = torch.arange(nb, dtype=torch.int32, device="cuda") * cap
        pos = (ctx - 1).to(torch.int64)
        slots = base.to(torch.int64) + pos
        cs = L.rope_cos_sin_table(m.max_position, hd, m.rope_theta).cuda()
        out = torch.empty(nb, nh * hd, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(L.attention_decode_workspace_size(nb, cap, nh, hd), dtype=torch.uint8, device="cuda")
        for _ in range(args.profile_reps):
            L.attention_decode_rope(qkv, nh, nkv, hd, m.tp, pos, cs, gamma, gamma, m.eps, slots, kc, vc, None, ctx,
                                    base, cap, hd ** -0.5, out, ws)
    if args.profile_kernel == "prefill.gemm_gate_up_silu":   # merged gate_up + SiluAndMul over the prompt tokens
        T, H, I = sum(seqs), m.hidden, m.intermediate
        x = rnd(T, H)
        w = (rnd(2 * I, H) * 0.02).to(torch.bfloat16)
        act = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(max(L.gemm_workspace_size(T, 2 * I, H, m.tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL,
                                                   torch.bfloat16), 16), dtype=torch.uint8, device="cuda")
        for _ in range(args.profile_reps):
            L.gemm(x, w, act, 2 * I, m.tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL, ws)
    torch.cuda.synchronize()
    L.device_error()


def main(argv=None):
    args = parse_args(argv)
    if args.profile_kernel is not None:
        profile_kernel(args)
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
