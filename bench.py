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
import itertools
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
    ap.add_argument("--profile-kernel", choices=["decode.attention", "decode.gemm_down", "prefill.gemm_gate_up_silu",
                                                 "prefill.attention"],
                    default=None,
                    help="launch only this kernel, --profile-reps times, on inputs of the workload's shape "
                         "(random values, mean decode context) and exit: a small case for ncu section captures")
    ap.add_argument("--profile-reps", type=int, default=3)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload lines (embedding + lm_head, one layer, 64-sequence decode)")
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
            "prefill.gemm_qkv_norm_rope_store_kv": ("tensor", 2.0 * T * qkvw * H),
            "prefill.gemm_o": ("tensor", 2.0 * T * H * nh * hd),
            "prefill.gemm_o_add_rmsnorm": ("tensor", 2.0 * T * H * nh * hd),
            "prefill.gemm_down_add_rmsnorm": ("tensor", 2.0 * T * H * I),
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
            # each launch: its ids, the table rows they select, the output rows
            "prefill.embed_vocab": ("hbm", 2.0 * 2 * T * H + 8.0 * T),
            "decode.embed_vocab": ("hbm", 2.0 * 2 * B * H + 8.0 * B),
        }

    def launches_per_step(self, kind):
        nl = self.m.n_layers
        fused_norm = self.fwd.norm_fusion_ok(self.B)
        if kind == "prefill.add_rmsnorm" and self.fwd.prefill_fusion_ok():
            return 1   # before the first layer; the o_proj / down epilogues do the rest
        per_layer = {"add_rmsnorm": 0 if fused_norm and kind.startswith("decode.") else 2}
        base = kind.split(".", 1)[-1]
        if kind == "lm_head":
            return 1 + self.S
        if kind == "prefill.embed_vocab":
            return 1
        if kind == "decode.embed_vocab":
            return self.S
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


def profile_traffic(name: str):
    """DRAM bytes per launch of a kernel from its committed ncu capture
    (profiles/<name>.json), or None when a source file it records has changed
    since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name + ".json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        prof = json.load(f)
    for rel, sha in prof.get("sources_sha1", {}).items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha1(f.read()).hexdigest() != sha:
                    return None
        except OSError:
            return None
    return prof.get("dram_bytes_per_launch")


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
    traffic = profile_traffic("decode_attention_bench_shape")
    if traffic is not None:   # the capture ran at the mean context: scale to this one
        traffic = round(traffic * sum(ctx) / (B * (statistics.mean(wl.seq_lens) + wl.S // 2)))
    return {"kernel": "decode.attention", "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 3), "traffic": traffic,
            "algorithmic_bytes": round(algo), "us_per_launch": round(us, 2),
            "peak_source": f"{peaks['source']} (HBM copy)",
            "timing": f"{m.n_layers} back-to-back launches over the {m.n_layers} layers' KV caches (larger than L2), "
                      f"decode step {s}, one CUDA graph replayed {reps} times, events on the replay stream"}


# ----------------------------------------------------------------------------
# the other workloads: one line each, with its own roofline
# ----------------------------------------------------------------------------

def _time_launches(fn, reps, flush=None):
    """Mean ms of fn() over reps launches, each timed alone with CUDA events on the
    current stream; flush() (an L2-sized write) runs before each, outside the events."""
    total = 0.0
    for _ in range(reps):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    return total / reps


def _graph(fn):
    fn()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        fn()
    torch.cuda.synchronize()
    return g


def _roof(bound, amount, ms, peaks, peak_key, what):
    if bound == "hbm":
        achieved, peak, unit = amount / (ms / 1e3) / 1e9, peaks["hbm"], "GB/s"
    else:
        achieved, peak, unit = amount / (ms / 1e3) / 1e12, peaks[peak_key], "TFLOP/s"
    return {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 3), "algorithmic": round(amount), "what": what,
            "peak_source": f"{peaks['source']} ({'HBM copy' if bound == 'hbm' else peak_key.replace('_', ' ')})"}


def config_embed_lm_head(peaks, reps=10):
    """Vocab-sharded embedding of 8192 ids (5 % on shard boundaries) and the lm_head
    producing the full [8192, 151936] logits, bf16, vocab 151936 x 1024."""
    import seeded_inputs as si
    from qwen3_transformer_forward_gb300 import _lib as L
    w = si.workload("embed_lm_head")
    m = w.model
    T, H, V = w.n_tokens, m.hidden, m.vocab
    table = si.checkpoint_tensor(m, "embed_tokens", device="cuda")
    ids = si.embed_ids(m, T, w.boundary_fraction).cuda()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # 256 MB > L2
    flush = flush_buf.zero_
    out = {}
    # the embedding: 16 launches back to back in one graph, each over its own id set (16 x 16.8 MB
    # of rows, more than L2 holds), so neither launch latency nor L2 hits enter the per-launch time
    R = 16
    id_sets = [ids] + [si.embed_ids(m, T, w.boundary_fraction, seed=1 + r).cuda() for r in range(R - 1)]
    embs = [torch.empty(T, H, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    for tp in w.tps:
        g = _graph(lambda: [L.embed_vocab(id_sets[r], table, tp, embs[r]) for r in range(R)])
        flush()
        ms = _time_launches(g.replay, 3, flush) / R
        out[f"embed_tp{tp}"] = {"us_per_launch": round(ms * 1e3, 2),
                                "roofline": _roof("hbm", 2.0 * 2 * T * H + 8.0 * T, ms, peaks, "hbm",
                                                  "ids + selected table rows + output rows")}
    del embs
    hidden = si.normal(0, "embed_lm_head.hidden", (T, H), 1.0, "bf16").cuda()
    logits = torch.empty(T, V, dtype=torch.bfloat16, device="cuda")
    for tp in w.tps:
        ws = torch.zeros(L.lm_head_workspace_size(T, V, H, tp, torch.bfloat16), dtype=torch.uint8, device="cuda")
        ms = _time_launches(lambda: L.lm_head(hidden, None, T, table, tp, logits, None, ws), max(3, reps // 2), flush)
        out[f"lm_head_tp{tp}"] = {"us_per_launch": round(ms * 1e3, 2),
                                  "roofline": _roof("tensor", 2.0 * T * H * V, ms, peaks, "tensor_burst",
                                                    "2 x 8192 x 1024 x 151936 FLOP (2.49 GB of logits written)")}
    L.device_error()
    del table, logits, flush_buf
    torch.cuda.empty_cache()
    return {"workload": "vocab 151936 x 1024 bf16, 8192 ids (5 % at shard boundaries), tp 1/2/4; "
                        "lm_head over 8192 N(0,1) hidden rows -> full [8192, 151936] logits",
            "timing": f"embedding: {R} launches back to back in a CUDA graph, each over its own 8192 ids (rows "
                      f"larger than L2 together), 3 replays after an L2 flush; lm_head: each launch alone after a "
                      f"256 MB L2 flush, CUDA events, mean of {max(3, reps // 2)}", **out}


def config_layer_prefill(peaks, reps=20):
    """One Qwen3-0.6B decoder layer, two shards, prefill of 4 x 512 tokens."""
    import seeded_inputs as si
    from qwen3_transformer_forward_gb300 import _lib as L
    from qwen3_transformer_forward_gb300 import model as M
    w = si.workload("layer_prefill")
    m = w.model
    b = si.prefill_batch(m, w.seq_lens)
    T = b.ids.shape[0]
    x = si.normal(0, "layer_prefill.hidden", (T, m.hidden), 1.0, "bf16").cuda()
    params = M.load_params(m, device="cuda")
    fwd = M.Qwen3Forward(m, params, max_tokens=T, num_slots=b.num_slots, max_seqs=len(w.seq_lens),
                         max_context=max(w.seq_lens))
    ctx = M.to_device_prefill(b)
    g = _graph(lambda: fwd.run_layers(ctx, decode=False, hidden_in=x, final_norm=False))
    ms = _time_launches(g.replay, reps)
    L.device_error()
    H, I, hd, nh, nkv = m.hidden, m.intermediate, m.head_dim, m.n_heads, m.n_kv_heads
    flops = 2.0 * T * ((nh + 2 * nkv) * hd * H + H * nh * hd + 2 * I * H + H * I) + \
        4.0 * hd * nh * sum(L_ * (L_ + 1) // 2 for L_ in w.seq_lens)
    return {"workload": "one Qwen3-0.6B layer (bf16, tp=2 layout), prefill 4 x 512, N(0,1) hidden inputs",
            "metric": "prefill tokens/s", "value": round(T / (ms / 1e3), 1), "unit": "tokens/s",
            "us_per_layer": round(ms * 1e3, 2),
            "roofline": _roof("tensor", flops, ms, peaks, "tensor_burst",
                              "GEMM + causal attention FLOP of the layer (68.7 GFLOP); the norms, RoPE and KV "
                              "store are HBM-bound extras inside the same time"),
            "timing": f"one CUDA graph of the layer's kernels (plus a 4 MB copy of the input rows), "
                      f"mean of {reps} replays; weights and activations fit in L2"}


def config_model_decode(peaks, reps=10):
    """The 28-layer model (tp 1), one decode step of 64 sequences with contexts
    uniform in [256, 2048] over a synthetic cache history."""
    import seeded_inputs as si
    from qwen3_transformer_forward_gb300 import _lib as L
    from qwen3_transformer_forward_gb300 import model as M
    w = si.workload("model_decode")
    m = w.model
    ctx_lens = si.decode_context_lens(0, w.batch, w.ctx_low, w.ctx_high)
    batch = si.decode_batch(m, ctx_lens)
    params = M.load_params(m, device="cuda")
    kc = [torch.zeros(batch.num_slots, m.n_kv_heads, m.head_dim, dtype=torch.bfloat16, device="cuda")
          for _ in range(m.n_layers)]
    vc = [torch.zeros_like(kc[0]) for _ in range(m.n_layers)]
    hist = torch.cat([torch.arange(int(batch.seq_base[b]), int(batch.seq_base[b]) + ctx_lens[b] - 1)
                      for b in range(w.batch)]).cuda()
    for l in range(m.n_layers):
        kc[l][hist] = si.kv_history(m, l, "k", hist)
        vc[l][hist] = si.kv_history(m, l, "v", hist)
    fwd = M.Qwen3Forward(m, params, max_tokens=w.batch, num_slots=batch.num_slots, max_seqs=w.batch,
                         max_context=max(ctx_lens), kv_caches=(kc, vc))
    ctx = M.to_device_decode(batch)
    g = _graph(lambda: fwd.decode(ctx))
    for _ in range(3):
        g.replay()
    ms = _time_launches(g.replay, reps)
    L.device_error()
    H, I, hd, nh, nkv, V = m.hidden, m.intermediate, m.head_dim, m.n_heads, m.n_kv_heads, m.vocab
    weights = m.n_layers * 2.0 * ((nh + 2 * nkv) * hd * H + H * nh * hd + 2 * I * H + H * I) + 2.0 * V * H
    kv = m.n_layers * 2.0 * 2 * nkv * hd * sum(ctx_lens)
    out = {"workload": "28-layer Qwen3-0.6B shape (bf16, tp=1), one decode step for 64 sequences, contexts "
                       "U[256, 2048] (sum %d) over a seeded N(0,1) cache history, greedy argmax" % sum(ctx_lens),
           "metric": "decode tokens/s", "value": round(w.batch / (ms / 1e3), 1), "unit": "tokens/s",
           "ms_per_step": round(ms, 3),
           "roofline": _roof("hbm", weights + kv, ms, peaks, "hbm",
                             f"every weight byte once ({weights / 1e9:.3f} GB incl. the tied table) + the cached "
                             f"K/V each sequence attends to ({kv / 1e9:.2f} GB)"),
           "timing": f"one CUDA graph of the step (embedding, 28 layers, final norm, lm_head, argmax), "
                     f"mean of {reps} replays after 3; {(weights + kv) / 1e9:.1f} GB streamed, larger than L2"}
    del fwd, kc, vc, params
    torch.cuda.empty_cache()
    return out


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
    launches = count_launches(wl)

    # the decode phase as a whole against HBM: every weight byte and the cached
    # K/V rows once per step, over the measured decode time (launch gaps,
    # phase boundaries and all)
    m = wl.m
    H, I, hd, nh, nkv, V = m.hidden, m.intermediate, m.head_dim, m.n_heads, m.n_kv_heads, m.vocab
    layer_w = 2.0 * ((nh + 2 * nkv) * hd * H + H * nh * hd + 2 * I * H + H * I)
    mean_ctx = statistics.mean(L0 + s + 1 for s in range(wl.S) for L0 in wl.seq_lens)
    layer_kv = 2.0 * 2 * nkv * hd * wl.B * mean_ctx
    step_bytes = m.n_layers * (layer_w + layer_kv) + 2.0 * V * H
    step_ms = decode_ms / wl.S
    decode_chain = {"bound": "hbm", "bytes_per_step": round(step_bytes), "ms_per_step": round(step_ms, 4),
                    "achieved": round(step_bytes / (step_ms / 1e3) / 1e9, 1), "peak": peaks["hbm"], "unit": "GB/s",
                    "frac": round(step_bytes / (step_ms / 1e3) / 1e9 / peaks["hbm"], 3),
                    "bytes_per_layer": round(layer_w + layer_kv),
                    "what": "28 layers' weights + the K/V each sequence attends to (mean context) + the tied "
                            "table for the lm_head, over the measured decode time per step"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)

    configs = None
    if not args.no_configs and world == 1:
        configs = {"embed_lm_head": config_embed_lm_head(peaks), "layer_prefill": config_layer_prefill(peaks),
                   "model_decode": config_model_decode(peaks)}


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
        "roofline": roofline, "decode_chain": decode_chain, "kernels": kernels, "clocks": clocks, "e2e": e2e,
        "cpu_baseline": cpu, "gpu_launches": launches, "configs": configs,
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
    if wl.fwd.prefill_fusion_ok():
        # embed, one add+RMSNorm, 5 per layer (QKV + norm/RoPE/KV store, attention, o_proj + add + norm,
        # gate_up + SiluAndMul, down + add + norm), gather + gemm + argmax
        prefill = 1 + 1 + m.n_layers * 5 + 3
    elif wl.fwd.qkv_epilogue_ok():
        prefill -= m.n_layers   # the QK-norm + RoPE + KV store runs in the QKV GEMM's epilogue
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


def cpu_sample_run(m, weights, cos_sin, n_tokens: int, decode_seqs: int = 8):
    """One bounded sample of the workload through the oracle:
      prefill: one sequence of n_tokens through the sampled layers, final norm and
               the lm_head of its last token;
      decode:  one decode step of decode_seqs sequences at context n_tokens + 1
               through the same layers (each sequence's cache holds the prefill's
               rows), final norm, lm_head and argmax of every sequence.
    Returns measured seconds and the full-model projection (layer time x
    n_layers / sampled layers)."""
    import numpy as np
    import oracle as O
    import seeded_inputs as si
    nl = len(weights.layers)
    b = si.prefill_batch(m, [n_tokens])
    cache = O.KVCache(nl, n_tokens, m.n_kv_heads, m.head_dim, m.tp)
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
    prefill_model = (t1 - t0) + (t2 - t1) * m.n_layers / nl + (t3 - t2)
    # decode: every sequence's cache = the prefill's rows, then this step's row
    L = n_tokens + 1
    dcache = O.KVCache(nl, decode_seqs * L, m.n_kv_heads, m.head_dim, m.tp)
    for r in range(m.tp):
        for l in range(nl):
            for q in range(decode_seqs):
                dcache.k[r][l][q * L:q * L + n_tokens] = cache.k[r][l]
                dcache.v[r][l][q * L:q * L + n_tokens] = cache.v[r][l]
    base = np.arange(decode_seqs) * L
    pos = np.full(decode_seqs, n_tokens)
    dctx = O.AttnContext(False, base + n_tokens, seq_base=base, context_lens=pos + 1)
    ids = si.uniform_int(0, "decode.forced_ids", (decode_seqs,), 0, m.vocab).numpy()
    t4 = time.perf_counter()
    h = O.vocab_parallel_embedding(ids, weights.embed, m.tp)
    t5 = time.perf_counter()
    res = None
    for l in range(nl):
        h, res = O.decoder_layer(m, weights.layers[l], l, pos, h, res, dctx, dcache, *cos_sin)
    t6 = time.perf_counter()
    h, _ = O.add_rms_norm(h, res, weights.final_norm, m.eps, m.dtype)
    O.greedy(O.compute_logits(m, weights.embed, h, m.tp))
    t7 = time.perf_counter()
    decode_model = (t5 - t4) + (t6 - t5) * m.n_layers / nl + (t7 - t6)
    return {"prefill_s": prefill_model, "decode_s": decode_model, "wall_s": (t3 - t0) + (t7 - t4)}


def cpu_projection(m, r, w):
    """Full-workload tokens/s from one sample: the step's prefill sequences each cost
    one sampled prefill, its decode steps each one sampled decode step."""
    n_seq, S, B = len(w.seq_lens), w.decode_steps, len(w.seq_lens)
    step_s = n_seq * r["prefill_s"] + S * r["decode_s"]
    tokens = sum(w.seq_lens) + S * B
    return tokens / step_s, step_s


def _cpu_sample_text(args, m, w):
    return (f"prefill of 1 sequence x {args.cpu_sample_tokens} tokens and one decode step of {len(w.seq_lens)} "
            f"sequences at context {args.cpu_sample_tokens + 1}, each through {args.cpu_sample_layers} of the "
            f"{m.n_layers} layers plus embedding, final norm and lm_head; layer time scaled x "
            f"{m.n_layers}/{args.cpu_sample_layers}; the workload step = {len(w.seq_lens)} such prefills + "
            f"{w.decode_steps} such decode steps (numpy float64, threads = all host cores)")


def cpu_baseline(args):
    import seeded_inputs as si
    m, weights, cos_sin = cpu_sample_setup(args.cpu_sample_layers)
    w = si.workload(WORKLOAD)
    r = cpu_sample_run(m, weights, cos_sin, args.cpu_sample_tokens)
    value, step_s = cpu_projection(m, r, w)
    return {"value": round(value, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "prefill_tok_s": round(args.cpu_sample_tokens / r["prefill_s"], 2),
            "decode_tok_s": round(len(w.seq_lens) / r["decode_s"], 3),
            "projected_step_s": round(step_s, 1), "sample_wall_s": round(r["wall_s"], 2),
            "sample": _cpu_sample_text(args, m, w)}


def run_reference(args, rank, world):
    import seeded_inputs as si
    if rank != 0:
        return None
    m, weights, cos_sin = cpu_sample_setup(args.cpu_sample_layers)
    w = si.workload(WORKLOAD)
    n = args.cpu_sample_tokens
    for _ in range(args.warmup):
        cpu_sample_run(m, weights, cos_sin, n)
    runs = [cpu_sample_run(m, weights, cos_sin, n) for _ in range(args.steps)]
    wall_ms = statistics.mean(r["wall_s"] for r in runs) * 1e3
    proj = [cpu_projection(m, r, w) for r in runs]
    value = statistics.mean(p[0] for p in proj)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall_ms, 1),
            "projected_ms_per_full_step": round(statistics.mean(p[1] for p in proj) * 1e3, 1),
            "prefill_tok_s": round(statistics.mean(n / r["prefill_s"] for r in runs), 2),
            "decode_tok_s": round(statistics.mean(len(w.seq_lens) / r["decode_s"] for r in runs), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded), random-init weights",
            "config": {"workload": "qwen3-0.6b-shape 28 layers, tp=2 layout, prefill 8x2048 + 128 greedy decode "
                                   "steps x 8 (bounded CPU sample, see cpu_baseline.sample)"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "each step: " + _cpu_sample_text(args, m, w) +
                                       "; ms_per_step is the measured wall time of the sample, value the "
                                       "full-step projection"},
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
    if args.profile_kernel == "decode.gemm_down":   # the decode step's row-split down projection, one weight copy per launch
        H, I, tp = m.hidden, m.intermediate, m.tp
        act = rnd(nb, I)
        ws_ = [(rnd(H, I) * 0.02).to(torch.bfloat16) for _ in range(max(1, args.profile_reps))]   # [tp][H][I/tp] order
        h = torch.empty(nb, H, dtype=torch.bfloat16, device="cuda")
        gws = torch.zeros(max(L.gemm_workspace_size(nb, H, I, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE, torch.bfloat16),
                              16), dtype=torch.uint8, device="cuda")
        for r in range(args.profile_reps):
            L.gemm(act, ws_[r], h, H, tp, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE, gws)
    if args.profile_kernel == "prefill.gemm_gate_up_silu":   # merged gate_up + SiluAndMul over the prompt tokens
        T, H, I = sum(seqs), m.hidden, m.intermediate
        x = rnd(T, H)
        w = (rnd(2 * I, H) * 0.02).to(torch.bfloat16)
        act = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(max(L.gemm_workspace_size(T, 2 * I, H, m.tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL,
                                                   torch.bfloat16), 16), dtype=torch.uint8, device="cuda")
        for _ in range(args.profile_reps):
            L.gemm(x, w, act, 2 * I, m.tp, L.QW_GEMM_COLUMN, L.QW_EPI_SILU_MUL, ws)
    if args.profile_kernel == "prefill.attention":   # causal prefill over the prompts, keys from the cache
        T = sum(seqs)
        q = rnd(T, nh, hd)
        kc, vc = rnd(T, nkv, hd), rnd(T, nkv, hd)
        cu = torch.tensor([0] + list(itertools.accumulate(seqs)), dtype=torch.int32, device="cuda")
        out = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
        for _ in range(args.profile_reps):
            L.attention_prefill(q, kc, vc, cu, cu, cu[:-1].contiguous(), max(seqs), nh, nkv, hd, hd ** -0.5, out)
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
