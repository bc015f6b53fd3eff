"""Benchmark of the speculative-decoding verify step on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  Workloads:

  dense-8b-verify-k4 (default): the verify step of an 8B-class dense bf16 target (36
      layers, d 4096, 32/8 heads, head_dim 128, SwiGLU 12288, vocab 151936, RMSNorm, RoPE
      theta 1e6, random-init N(0, 0.02^2) weights), B = 1, a 1024-token random prompt,
      K = 4 drafts, greedy.  A scripted drafter copies j ~ Geometric(alpha 0.7) capped at K
      tokens of the target's own recorded greedy trajectory and then one wrong token.  A
      step is one spec_verify call: embed, 36 layers (RMSNorm, QKV GEMM + RoPE + KV append,
      paged attention, O GEMM + residual, RMSNorm, gate/up GEMM + SwiGLU, down GEMM +
      residual), final norm, lm_head, fused verify, KV trim.
  verify-logits-b64-k4: the fused verify kernel alone on fp32 logits, B = 64, K = 4,
      vocab 151936, temperature 1.0, top-k 20, top-p 0.95.
  sampling-27b-0p8b: a 27B-class bf16 target with a 0.8B-class bf16 draft, B = 1, a
      2048-token prompt, temperature 1.0, top-k 20, top-p 0.95; a step is one round of K = 4
      sampled drafts and the target's verify against the draft logits; a K sweep over
      {1, 2, 4, 8, 16} goes beside it.
  serving-8b-b32-k8: batched verify on the 8B-class shape, B = 32 sequences with KV
      lengths uniform in [2048, 16384], n-gram drafts (K = 8 with per-sequence draft
      lengths) from the drafter on the device, a KV trim after every step.

The metric is emitted tokens per second of verify steps (accepted drafts plus the
correction or bonus token); ms_per_step is the verify-step latency; `roofline` is the
achieved HBM bandwidth of the dominant kernel.
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

METRIC = "verify-step latency & HBM GB/s vs 8 TB/s peak; accepted tokens/s at fixed K"
VOCAB = 151936


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---- clocks -------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        self.lines = []

    def __enter__(self):
        import torch
        ident = None
        try:
            ident = str(torch.cuda.get_device_properties(self.dev).uuid)
            if not ident.startswith("GPU-"):
                ident = "GPU-" + ident
        except Exception:
            ident = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if ident:
            cmd += ["-i", ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- distributed plumbing ---------------------------------------------------------------

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- workload: the 8B verify step ---------------------------------------------------------

class DenseVerifyWorkload:
    name = "dense-8b-verify-k4"
    dtype = "bf16"

    def __init__(self, K=4, prompt_len=1024, alpha=0.7, n_gen=512, layers=None):
        import dataclasses
        import synth
        self.shape = synth.QWEN_8B
        if layers is not None and layers != self.shape.n_layers:
            # a slice of the 8B shape with fewer layers (small cases for profiler captures)
            self.shape = dataclasses.replace(self.shape, n_layers=layers, name=f"dense-8b-{layers}l")
        self.K, self.prompt_len, self.alpha, self.n_gen = K, prompt_len, alpha, n_gen

    def config(self):
        s = self.shape
        return {"workload": self.name,
                "model_shape": f"{s.n_layers} layers, d {s.d_model}, {s.n_q_heads}/{s.n_kv_heads} heads, head_dim "
                               f"{s.head_dim}, SwiGLU {s.ffn_dim}, vocab {s.vocab}, bf16, random init N(0,0.02^2)",
                "B": 1, "K": self.K, "prompt_len": self.prompt_len, "decoding": "greedy",
                "drafter": f"scripted: j~Geometric(acceptance {self.alpha}) capped at K true tokens of the "
                           "target's recorded greedy trajectory, then a wrong token",
                "l2": "inputs larger than L2 (15.1 GB of weights streamed per step)"}

    def setup(self, device, n_steps):
        import torch
        import synth
        from speculative_decoding_verify_token_gb300 import model as M, generate as G
        s, K = self.shape, self.K
        self.weights = synth.model_weights(s, seed=0, device=device)
        self.traj_len = max(self.n_gen, (K + 1) * n_steps + 8)
        max_ctx = self.prompt_len + self.traj_len + 64
        self.m = M.SpecModel(s, self.weights, max_batch=1, max_ctx=max_ctx, max_k=K, prefill_chunk=256)
        self.prompt = torch.from_numpy(synth.prompt_tokens(1, self.prompt_len, s.vocab)).to(device)
        traj = G.plain_generate(self.m, self.prompt, self.traj_len)
        self.seq = torch.cat([self.prompt, traj]).cpu().numpy()
        g = np.random.Generator(np.random.PCG64(4))
        pos = self.prompt_len - 1
        last, drafts, js, nexts = [], [], [], []
        for _ in range(n_steps):
            j = min(int(g.geometric(1.0 - self.alpha)) - 1, K)
            d = [int(self.seq[pos + 1 + i]) for i in range(j)]
            while len(d) < K:
                true = int(self.seq[pos + 1 + len(d)])
                d.append(int((true + 1 + g.integers(0, s.vocab - 1)) % s.vocab))
            last.append(int(self.seq[pos]))
            drafts.append(d)
            js.append(j)
            nexts.append(int(self.seq[pos + j + 1]))
            pos += j + 1
        self.n_steps = n_steps
        self.js, self.nexts = np.array(js), np.array(nexts)
        self.d_last = torch.tensor(last, dtype=torch.int32, device=device).view(n_steps, 1)
        self.d_drafts = torch.tensor(drafts, dtype=torch.int32, device=device).view(n_steps, 1, K)
        self.d_u = torch.full((1, K + 1), 0.5, dtype=torch.float32, device=device)
        self.outs = [{"accepted_len": torch.empty(1, dtype=torch.int32, device=device),
                      "next_token": torch.empty(1, dtype=torch.int32, device=device),
                      "out_ids": torch.empty(1, 32, dtype=torch.int32, device=device),
                      "out_probs": torch.empty(1, 32, dtype=torch.float32, device=device),
                      "status": torch.empty(1, dtype=torch.int32, device=device)} for _ in range(n_steps)]
        self.reset()
        torch.cuda.synchronize()

    def reset(self):
        self.m.reset(0)
        self.m.prefill(0, self.prompt[:-1])

    def step(self, i):
        self.m.verify([0], self.d_last[i], self.d_drafts[i], self.d_u, 0.0, out=self.outs[i])

    def launches(self):
        return self.m.launches()

    def check(self, i0, n):
        """Every timed step must accept exactly the scripted j and emit the trajectory token."""
        a = np.array([int(self.outs[i]["accepted_len"].item()) for i in range(i0, i0 + n)])
        nx = np.array([int(self.outs[i]["next_token"].item()) for i in range(i0, i0 + n)])
        ok = bool(np.all(a == self.js[i0:i0 + n]) and np.all(nx == self.nexts[i0:i0 + n]))
        return ok, int(a.sum() + n)

    def decode_ms(self, n):
        """Single-token decode step on the same context (the comparator of the verify step)."""
        import torch
        self.reset()
        tok = self.d_last[0][0:1].clone()
        outs = [torch.empty(1, dtype=torch.int32, device=tok.device) for _ in range(n + 3)]
        for i in range(3):
            tok = self.m.decode([0], tok, out=outs[i])
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            tok = self.m.decode([0], tok, out=outs[3 + i])
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    def profile(self, n):
        self.reset()
        self.m.profile(True)
        for i in range(n):
            self.step(i)
        prof = self.m.profile_read()
        self.m.profile(False)
        return prof

    def roofline(self, prof, peaks, ms_per_step=None, profile_steps=1):
        """The graphed verify step as the unit: its algorithmic bytes (the weights of every GEMM,
        the KV pages read and written, the logits) over the timed step's CUDA-event time."""
        step_bytes = sum(v["bytes"] for v in prof.values()) / profile_steps
        achieved = step_bytes / (ms_per_step / 1e3) / 1e9
        L = self.shape.n_layers
        # DRAM bytes (read + write) of every kernel of one graphed verify step, from an ncu
        # capture of a 2-layer slice of this shape (--cache-control none), scaled to L layers
        # by the per-layer share (every layer moves the same weights); None until re-taken
        # after a change to the kernels
        traffic = (L * STEP_TRAFFIC_PER_LAYER + STEP_TRAFFIC_FIXED) if STEP_TRAFFIC_PER_LAYER else None
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": f"verify step: the graphed pass ({4 * L + 1} tc_gemm_kernel, {L} attention + "
                          f"{L} combine, embed, 2 verify, length update)",
                "traffic_unit": "bytes per step", "algorithmic_bytes_per_launch": step_bytes,
                "avg_launch_us": ms_per_step * 1e3, "launch_unit": "one graphed verify step",
                "peak_source": peaks["source"]}

    # end to end through the C ABI with host buffers
    def e2e(self, n):
        import torch
        self.reset()
        h_last = self.d_last.cpu().pin_memory()
        h_drafts = self.d_drafts.cpu().pin_memory()
        h_u = self.d_u.cpu().pin_memory()
        d_last = torch.empty(1, dtype=torch.int32, device="cuda")
        d_drafts = torch.empty(1, self.K, dtype=torch.int32, device="cuda")
        d_u = torch.empty(1, self.K + 1, dtype=torch.float32, device="cuda")
        h_out = torch.empty(2, dtype=torch.int32).pin_memory()
        st = torch.cuda.current_stream()
        emitted = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            d_last.copy_(h_last[i].view(1), non_blocking=True)
            d_drafts.copy_(h_drafts[i], non_blocking=True)
            d_u.copy_(h_u, non_blocking=True)
            o = self.m.verify([0], d_last, d_drafts, d_u, 0.0, out=self.outs[i])
            h_out[0:1].copy_(o["accepted_len"], non_blocking=True)
            h_out[1:2].copy_(o["next_token"], non_blocking=True)
            st.synchronize()
            emitted += int(h_out[0]) + 1
        dt = time.perf_counter() - t0
        return emitted / dt, 4 + 4 * self.K + 4 * (self.K + 1), 8

    def oracle_sample(self, budget_s):
        """The float64 oracle timed on the same verify step as the GPU's (dense_oracle_step):
        as many whole steps as fit the budget (at least one)."""
        step, sample = dense_oracle_step(self.shape, self.K, self.alpha)
        n, t0 = 0, time.perf_counter()
        emitted = 0.0
        while n == 0 or time.perf_counter() - t0 < budget_s:
            emitted += step()
            n += 1
        return emitted / (time.perf_counter() - t0), f"{n} step(s): " + sample


def dense_oracle_step(shape, K, alpha):
    """One float64 oracle verify step of the 8B workload, for the CPU baseline and the
    reference arm: the verify pass of K + 1 tokens through all L layers at a context of 63
    tokens (every layer uses layer 0's weights, generated once, so that the weights held on
    the host stay at one layer's; the cost per layer is the same), the full-vocabulary
    lm_head and the greedy rule; no prefill inside the step.  The scripted drafter's
    decisions need the real model, so a step counts the closed-form mean of
    (1 - alpha^(K+1)) / (1 - alpha) emitted tokens."""
    import copy
    from synth import fastgen
    from oracle import model as om
    from oracle import verify as ov
    import synth
    held = {}

    def w(name):
        base = name if not name.startswith("layers.") else "layers.0." + name.split(".", 2)[2]
        if base not in held:
            held[base] = fastgen.EmbedRowsF64(shape) if base == "embed" else fastgen.model_weight_f64(shape, base)
        return held[base]

    dec = om.Decoder(shape, w)
    cache0 = dec.new_cache()
    dec.forward(synth.prompt_tokens(1, 63, shape.vocab), cache0, logits_rows=np.zeros(0, dtype=np.int64))
    toks = [int(t) for t in synth.prompt_tokens(2, K + 1, shape.vocab)]
    per_step = (1 - alpha ** (K + 1)) / (1 - alpha)

    def step():
        cache = copy.deepcopy(cache0)
        rows = dec.forward(toks, cache)
        ov.verify_greedy(rows, toks[1:])
        return per_step

    return step, (f"float64 oracle verify pass of {K + 1} tokens through {shape.n_layers} layers (context 63, every "
                  f"layer with layer 0's weights) + the {shape.vocab}-row lm_head + the greedy rule, no prefill in "
                  f"the step; {per_step:.4f} emitted tokens per step (closed form at acceptance {alpha})")


# ---- workload: 27B target + 0.8B draft under sampling -------------------------------------

class SamplingWorkload:
    """A 27B-class bf16 target with a 0.8B-class bf16 draft, B = 1, a 2048-token prompt,
    temperature 1, top-k 20, top-p 0.95 on both sides.  A step is one speculative round at
    K = 4: the draft decodes K tokens one at a time, each sampled from its truncated q with
    a seeded uniform, then the target verifies them in one pass against the draft logits
    (rejection sampling with the same truncation), and both caches are trimmed.  The round
    reads the accepted length back (the next round's draft input depends on it), so the
    value is emitted tokens over the rounds' span, drafting included.  `k_sweep` repeats
    the generation of 512 tokens for K in {1, 2, 4, 8, 16} from the same prefilled prompt."""
    name = "sampling-27b-0p8b"
    dtype = "bf16"

    def __init__(self, K=4, prompt_len=2048, n_sweep=512, sweep=(1, 2, 4, 8, 16), layers=None, **_):
        import dataclasses
        import synth
        self.shape, self.dshape = synth.QWEN_27B, synth.DRAFT_0P8B
        if layers is not None and layers != self.shape.n_layers:
            self.shape = dataclasses.replace(self.shape, n_layers=layers, name=f"dense-27b-{layers}l")
        self.K, self.prompt_len, self.n_sweep, self.sweep = K, prompt_len, n_sweep, tuple(sweep)
        self.T, self.k, self.p = 1.0, 20, 0.95

    def config(self):
        s, d = self.shape, self.dshape
        return {"workload": self.name,
                "model_shape": f"target {s.n_layers} layers, d {s.d_model}, {s.n_q_heads}/{s.n_kv_heads} heads, "
                               f"head_dim {s.head_dim}, SwiGLU {s.ffn_dim}; draft {d.n_layers} layers, d {d.d_model}, "
                               f"{d.n_q_heads}/{d.n_kv_heads} heads, SwiGLU {d.ffn_dim}; vocab {s.vocab}, bf16, "
                               "random init N(0,0.02^2)",
                "B": 1, "K": self.K, "prompt_len": self.prompt_len, "decoding": "sampling T 1.0, top-k 20, top-p 0.95",
                "uniforms": "verify PCG64 seed 2, draft PCG64 seed 4",
                "l2": "inputs larger than L2 (target weights streamed per verify, draft weights per draft token)"}

    def setup(self, device, n_steps):
        import torch
        import synth
        from speculative_decoding_verify_token_gb300 import model as M
        self.dev = device
        self.wt = synth.model_weights(self.shape, seed=0, device=device)
        self.wd = synth.model_weights(self.dshape, seed=0, device=device)
        kmax = max((self.K,) + self.sweep)
        max_ctx = self.prompt_len + max(self.n_sweep, (self.K + 1) * n_steps) + 8 * (kmax + 1) + 64
        self.t = M.SpecModel(self.shape, self.wt, max_ctx=max_ctx, max_k=kmax, prefill_chunk=256)
        self.d = M.SpecModel(self.dshape, self.wd, max_ctx=max_ctx, max_k=kmax, prefill_chunk=256)
        self.prompt = torch.from_numpy(synth.prompt_tokens(1, self.prompt_len, self.shape.vocab)).to(device)
        self.log = []
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        self.reset()
        torch.cuda.synchronize()

    def reset(self):
        self.t.reset(0)
        self.d.reset(0)
        self.t.prefill(0, self.prompt[:-1])
        self.d.prefill(0, self.prompt[:-1])
        self.pending = self.prompt[-1:].clone()
        self.extra = None
        self.g = np.random.Generator(np.random.PCG64(2))
        self.gd = np.random.Generator(np.random.PCG64(4))

    def _round(self, K, u=None, ud=None):
        import torch
        dev = self.dev
        e0, e1, e2 = self.ev
        e0.record()
        if self.extra is not None:
            self.d.prefill(0, self.extra)
        if ud is None:
            ud = torch.from_numpy(self.gd.random((1, K), dtype=np.float32)).to(dev, non_blocking=True)
        # the draft's K tokens in one device-resident loop (spec_draft, one graph per K)
        drafts, dl = self.d.draft([0], self.pending, K, ud.view(1, K), self.T, self.k, self.p, want_logits=True)
        if u is None:
            u = torch.from_numpy(self.g.random((1, K + 1), dtype=np.float32)).to(dev, non_blocking=True)
        e1.record()
        r = self.t.verify([0], self.pending, drafts, u, self.T, self.k, self.p, draft_logits=dl)
        e2.record()
        a = int(r["accepted_len"].item())
        self.d.kv_trim([0], K - 1, torch.clamp(r["accepted_len"], max=K - 1))
        self.extra = drafts[0, K - 1:K].clone() if a == K else None
        self.pending = r["next_token"].clone()
        ok = int(r["status"].item()) == 0
        self.log.append((a + 1, K, a, ok, e0.elapsed_time(e1), e1.elapsed_time(e2)))

    def step(self, i):
        self._round(self.K)

    def launches(self):
        return self.t.launches() + self.d.launches()

    def check(self, i0, n):
        rows = self.log[i0:i0 + n]
        return all(r[3] for r in rows), int(sum(r[0] for r in rows))

    def stats(self, i0, n):
        rows = self.log[i0:i0 + n]
        return {"acceptance": sum(r[2] for r in rows) / max(1, sum(r[1] for r in rows)),
                "emitted_per_step": sum(r[0] for r in rows) / max(1, len(rows)),
                "draft_ms_per_step": sum(r[4] for r in rows) / max(1, len(rows)),
                "verify_ms_per_step": sum(r[5] for r in rows) / max(1, len(rows))}

    def k_sweep(self):
        """512 new tokens per K from the same prompt: accepted tokens/s over the decode wall
        time (drafting included), the verify pass's and the drafting's event times."""
        import torch
        out = {}
        for K in self.sweep:
            self.reset()
            torch.cuda.synchronize()
            i0 = len(self.log)
            emitted = 0
            t0 = time.perf_counter()
            while emitted < self.n_sweep:
                self._round(K)
                emitted += self.log[-1][0]
            dt = time.perf_counter() - t0
            st = self.stats(i0, len(self.log) - i0)
            out[str(K)] = {"tokens_per_s": emitted / dt, "rounds": len(self.log) - i0, **st}
        return out

    def profile(self, n):
        self.t.profile(True)
        for _ in range(n):
            self._round(self.K)
        prof = self.t.profile_read()
        self.t.profile(False)
        return prof

    def roofline(self, prof, peaks):
        g = [prof[k] for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_lm_head")]
        ms = sum(x["ms"] for x in g)
        n = sum(x["launches"] for x in g)
        by = sum(x["bytes"] for x in g)
        achieved = (by / n) / (ms / n / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": "tc_gemm_kernel",
                "model": "target", "algorithmic_bytes_per_launch": by / n, "launches_measured": n,
                "avg_launch_us": ms / n * 1e3, "peak_source": peaks["source"]}

    def e2e(self, n):
        """The same rounds with the verify uniforms, the draft uniforms and the pending token
        taken from pinned host memory every round and the round's outputs read back."""
        import torch
        h_u = torch.from_numpy(self.g.random((n, self.K + 1), dtype=np.float32)).pin_memory()
        h_ud = torch.from_numpy(self.gd.random((n, self.K), dtype=np.float32)).pin_memory()
        torch.cuda.synchronize()
        emitted = 0
        t0 = time.perf_counter()
        for i in range(n):
            self._round(self.K, u=h_u[i:i + 1].to(self.dev, non_blocking=True),
                        ud=h_ud[i].to(self.dev, non_blocking=True))
            emitted += self.log[-1][0]
        dt = time.perf_counter() - t0
        return emitted / dt, 4 * (self.K + 1) + 4 * self.K, 8

    def oracle_sample(self, budget_s):
        """The float64 oracle on a bounded sample of one round: the target's verify pass of
        K + 1 tokens and the draft's K single-token passes, each through 1 layer (context 63)
        with a 4096-row lm_head slice, scaled to 64 and 28 layers and the full vocabulary, at
        the measured emitted tokens per round."""
        import dataclasses
        import synth
        from oracle import model as om
        out_t = []
        for shp, n_tok, passes in ((self.shape, self.K + 1, 1), (self.dshape, 1, self.K)):
            sub = dataclasses.replace(shp, n_layers=1, vocab=4096)
            names = [n for n in synth.weight_names(sub) if n.startswith("layers.0.")]
            w = {n: om.to_f64(synth.model_weight(shp, n, seed=0)) for n in names}
            w["embed"] = om.to_f64(synth.model_weight(sub, "embed", seed=0))
            w["final_norm"] = np.ones(shp.d_model)
            w["lm_head"] = om.to_f64(synth.model_weight(sub, "lm_head", seed=0))
            dec = om.Decoder(sub, w)
            cache = dec.new_cache()
            dec.forward(synth.prompt_tokens(1, 63, sub.vocab), cache)
            toks = [int(t) for t in synth.prompt_tokens(2, n_tok, sub.vocab)]
            t0 = time.perf_counter()
            dec.forward(toks, cache)
            dt = time.perf_counter() - t0
            out_t.append(dt * shp.n_layers * shp.vocab / sub.vocab * passes)
        st = self.stats(0, len(self.log))
        return st["emitted_per_step"] / sum(out_t), (
            f"float64 target pass of {self.K + 1} tokens and {self.K} draft single-token passes, each through 1 "
            f"layer (context 63) with a 4096-row lm_head slice, scaled to {self.shape.n_layers}/"
            f"{self.dshape.n_layers} layers and the full vocabulary, at {st['emitted_per_step']:.3f} emitted tokens "
            "per round")


# ---- workload: batched serving with an n-gram drafter -----------------------------------

class ServingWorkload:
    """Batched serving verify on the 8B shape: B sequences with ragged prompt lengths
    U[len_lo, len_hi] built from spans of which 40% copy an earlier window of the same
    sequence; drafts from the n-gram drafter on the device (longest suffix match of 8 down to
    3 tokens, at most K tokens, draft_len per sequence) over each slot's recorded tokens;
    greedy verify with auto trim.  A step is one serving round: spec_ngram_draft_device,
    spec_verify (pending tokens, drafts and draft lengths stay on the device between them)
    and the download of drafts, accepted lengths, next tokens and draft lengths (the emitted
    tokens are drafts[:accepted] + next).  Drafting + verify are timed with CUDA events on
    the stream (value, ms_per_step); the whole round is the end-to-end number."""
    name = "serving-8b-b32-k8"
    dtype = "bf16"
    device_timed = True

    def __init__(self, B=32, K=8, len_lo=2048, len_hi=16384, layers=None, **_):
        import dataclasses
        import synth
        self.shape = synth.QWEN_8B
        if layers is not None and layers != self.shape.n_layers:
            self.shape = dataclasses.replace(self.shape, n_layers=layers, name=f"dense-8b-{layers}l")
        self.B, self.K, self.len_lo, self.len_hi = B, K, len_lo, len_hi

    def config(self):
        s = self.shape
        return {"workload": self.name,
                "model_shape": f"{s.n_layers} layers, d {s.d_model}, {s.n_q_heads}/{s.n_kv_heads} heads, head_dim "
                               f"{s.head_dim}, SwiGLU {s.ffn_dim}, vocab {s.vocab}, bf16, random init N(0,0.02^2)",
                "B": self.B, "K": self.K, "prompt_len": f"U[{self.len_lo}, {self.len_hi}] per sequence (seed 5)",
                "kv_tokens_at_start": int(self.lens.sum()) if hasattr(self, "lens") else None,
                "prompts": "spans of U[8,64] tokens, 40% copying an earlier window of the same sequence",
                "decoding": "greedy", "drafter": "n-gram lookup on the device, suffix match 8..3 tokens, <= K drafted",
                "kv_cache": "paged bf16, 16-token pages",
                "l2": "inputs larger than L2 (15.1 GB of weights + the KV cache streamed per step)"}

    def setup(self, device, n_steps):
        import torch
        import synth
        from speculative_decoding_verify_token_gb300 import model as M
        s, B, K = self.shape, self.B, self.K
        g = np.random.Generator(np.random.PCG64(5))
        self.lens = g.integers(self.len_lo, self.len_hi + 1, size=B)
        self.seq_ids = list(range(B))
        self.weights = synth.model_weights(s, seed=0, device=device)
        max_ctx = int(self.lens.max()) + (K + 1) * (n_steps + 64) + 64
        self.m = M.SpecModel(s, self.weights, max_batch=B, max_ctx=max_ctx, max_k=K, prefill_chunk=256)
        last = []
        for b in range(B):
            prompt = synth.ngram_prompt(5 + b, int(self.lens[b]), s.vocab)
            self.m.prefill(b, torch.from_numpy(prompt[:-1]).to(device))
            last.append(int(prompt[-1]))
        self.kv_len = self.lens.astype(np.int64) - 1        # committed tokens in each slot's cache
        self.pending = torch.tensor(last, dtype=torch.int32, device=device)
        self.h_out = torch.zeros(3, B, dtype=torch.int32).pin_memory()
        self.h_drafts = torch.zeros(B, K, dtype=torch.int32).pin_memory()
        self.d_drafts = torch.empty(B, K, dtype=torch.int32, device=device)
        self.d_len = torch.empty(B, dtype=torch.int32, device=device)
        self.d_u = torch.zeros(B, K + 1, dtype=torch.float32, device=device)
        self.out = {"accepted_len": torch.empty(B, dtype=torch.int32, device=device),
                    "next_token": torch.empty(B, dtype=torch.int32, device=device),
                    "out_ids": torch.empty(B, 32, dtype=torch.int32, device=device),
                    "out_probs": torch.empty(B, 32, dtype=torch.float32, device=device),
                    "status": torch.empty(B, dtype=torch.int32, device=device)}
        self.ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
        self.log = []              # per step: (emitted, drafted, accepted, status ok, kv tokens read)
        self.dev_ms = []
        torch.cuda.synchronize()

    def _round(self, timed_events=True):
        import torch
        B, K = self.B, self.K
        kv_read = int(self.kv_len.sum())
        a, b = self.ev[len(self.dev_ms) % len(self.ev)]
        a.record()
        self.m.ngram_draft(self.seq_ids, self.pending, K, 3, 8, out=(self.d_drafts, self.d_len))
        self.m.verify(self.seq_ids, self.pending, self.d_drafts, self.d_u, 0.0, draft_len=self.d_len, out=self.out)
        b.record()
        self.h_out[0].copy_(self.out["accepted_len"], non_blocking=True)
        self.h_out[1].copy_(self.out["next_token"], non_blocking=True)
        self.h_out[2].copy_(self.d_len, non_blocking=True)
        self.h_drafts.copy_(self.d_drafts, non_blocking=True)
        self.pending.copy_(self.out["next_token"])
        torch.cuda.current_stream().synchronize()
        self.dev_ms.append(a.elapsed_time(b))
        acc = self.h_out[0].numpy().astype(np.int64)
        nxt = self.h_out[1].numpy()
        lens = self.h_out[2].numpy().astype(np.int64)
        st_ok = bool(np.all((lens >= 0) & (lens <= K) & (acc >= 0) & (acc <= lens) & (nxt >= 0)
                            & (nxt < self.shape.vocab)))
        acc = np.clip(acc, 0, lens)
        self.kv_len += acc + 1
        self.log.append((int(acc.sum()) + B, int(lens.sum()), int(acc.sum()), st_ok, kv_read))

    def step(self, i):
        self._round()

    def launches(self):
        return self.m.launches()

    def check(self, i0, n):
        rows = self.log[i0:i0 + n]
        ok = all(r[3] for r in rows) and int(self.out["status"].abs().sum().item()) == 0
        return ok, int(sum(r[0] for r in rows))

    def timed_ms(self, i0, n):
        return float(sum(self.dev_ms[i0:i0 + n]))

    def stats(self, i0, n):
        rows = self.log[i0:i0 + n]
        drafted = sum(r[1] for r in rows)
        accepted = sum(r[2] for r in rows)
        kv = sum(r[4] for r in rows) / max(len(rows), 1)
        first = self.log[0]
        return {"acceptance": accepted / max(drafted, 1), "drafted_per_step": drafted / max(len(rows), 1),
                "emitted_per_step": sum(r[0] for r in rows) / max(len(rows), 1), "kv_tokens_per_step": kv,
                "first_round": {"drafted": first[1], "accepted": first[2]},
                "acceptance_note": "random-init weights: the first round drafts from the prompts' copied spans; "
                                   "once a sequence ends in tokens the model emitted, a random-init model's "
                                   "greedy tokens do not repeat its context, so no suffix of 3+ tokens recurs, "
                                   "the lookup drafts nothing and the round emits one token for that sequence "
                                   "(each round still verifies K+1 rows per sequence)"}

    def profile(self, n):
        self.m.profile(True)
        for _ in range(n):
            self._round()
        prof = self.m.profile_read()
        self.m.profile(False)
        return prof

    def roofline(self, prof, peaks):
        # the kernel class with the largest time share (attention at these context lengths)
        cls = max((k for k in prof if prof[k]["launches"] and k != "other"), key=lambda k: prof[k]["ms"])
        x = prof[cls]
        attn = "attn_tc_kernel + attn_combine128_kernel" if self.B > 4 else "attn_mma_kernel + attn_combine128_kernel"
        kernel = {"attention": attn, "verify": "verify_kernel"}.get(cls, "tc_gemm_kernel")
        achieved = (x["bytes"] / x["launches"]) / (x["ms"] / x["launches"] / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": kernel, "class": cls,
                "algorithmic_bytes_per_launch": x["bytes"] / x["launches"], "launches_measured": x["launches"],
                "avg_launch_us": x["ms"] / x["launches"] * 1e3, "peak_source": peaks["source"]}

    def e2e(self, n):
        """Serving rounds through the C ABI: drafting and verify on the device, then the
        download of the drafts, accepted lengths, next tokens and draft lengths (from which a
        server streams out drafts[:accepted] + next); nothing is uploaded per round."""
        import torch
        torch.cuda.synchronize()
        i0 = len(self.log)
        t0 = time.perf_counter()
        for _ in range(n):
            self._round()
        dt = time.perf_counter() - t0
        emitted = sum(r[0] for r in self.log[i0:])
        return emitted / dt, 0, 4 * self.B * (self.K + 3)

    def oracle_sample(self, budget_s):
        """The float64 oracle on a bounded sample: the verify pass of K+1 tokens of one
        sequence through 1 of the 36 layers at a context of 255 tokens, plus final norm and
        a 4096-row slice of lm_head; scaled to 36 layers, the full lm_head and B sequences,
        at the measured emitted tokens per step.  Attention over the real 2k-16k contexts is
        not scaled, so the oracle's rate is an upper bound."""
        import dataclasses
        import synth
        from oracle import model as om
        from oracle import verify as ov
        s = self.shape
        sub = dataclasses.replace(s, n_layers=1, vocab=4096)
        names = [n for n in synth.weight_names(sub) if n.startswith("layers.0.")]
        w = {n: om.to_f64(synth.model_weight(s, n, seed=0)) for n in names}
        w["embed"] = om.to_f64(synth.model_weight(sub, "embed", seed=0))
        w["final_norm"] = np.ones(s.d_model)
        w["lm_head"] = om.to_f64(synth.model_weight(sub, "lm_head", seed=0))
        dec = om.Decoder(sub, w)
        prompt = synth.ngram_prompt(5, 255, sub.vocab)
        toks = [int(t) for t in synth.prompt_tokens(2, self.K + 1, sub.vocab)]
        cache = dec.new_cache()
        dec.forward(prompt, cache)
        t0 = time.perf_counter()
        rows = dec.forward(toks, cache)
        ov.verify_greedy(rows, toks[1:])
        t_pass = time.perf_counter() - t0
        per_step = t_pass * s.n_layers * s.vocab / sub.vocab * self.B
        st = self.stats(0, len(self.log))
        return st["emitted_per_step"] / per_step, (
            f"float64 verify pass of {self.K + 1} tokens of 1 sequence through 1 of {s.n_layers} layers (context "
            f"255) + a 4096-row lm_head slice, scaled to {s.n_layers} layers, the full lm_head and {self.B} "
            f"sequences at {st['emitted_per_step']:.2f} emitted tokens per step; attention over the 2k-16k "
            f"contexts not scaled")


# ---- workload: standalone verify on logits ----------------------------------------------

class VerifyLogitsWorkload:
    name = "verify-logits-b64-k4"
    dtype = "f32"

    def __init__(self, B=64, K=4, V=VOCAB, T=1.0, top_k=20, top_p=0.95, seed=3):
        self.B, self.K, self.V, self.T, self.k, self.p, self.seed = B, K, V, T, top_k, top_p, seed

    def config(self):
        return {"workload": self.name, "B": self.B, "K": self.K, "vocab": self.V, "temperature": self.T,
                "top_k": self.k, "top_p": self.p, "logits": "fp32 N(0,3^2) + shared Gumbel-perturbed spike",
                "l2": "inputs larger than L2 (two 350 MB sets alternate)"}

    def bytes_per_step(self):
        return self.B * (2 * self.K + 1) * self.V * 4

    def setup(self, device, n_steps):
        import torch
        import synth
        from speculative_decoding_verify_token_gb300 import verify as sv
        self.sv = sv
        self.sets = []
        for s in range(2):
            case = synth.verify_logits_case(self.seed + s, self.B, self.K, self.V)
            tgt = torch.from_numpy(case["target"]).to(device)
            dft = torch.from_numpy(case["draft"]).to(device)
            ud = torch.from_numpy(case["u_draft"]).to(device).reshape(-1)
            drafts = sv.sample_logits(dft.view(-1, self.V), ud, self.T, self.k, self.p).view(self.B, self.K)
            u = torch.from_numpy(case["u"]).to(device)
            self.sets.append((tgt, dft, drafts, u, case))
        self.ws = sv.verify_workspace(self.B, self.K, self.V, device)
        self.outs = [{"accepted_len": torch.empty(self.B, dtype=torch.int32, device=device),
                      "next_token": torch.empty(self.B, dtype=torch.int32, device=device),
                      "out_ids": torch.empty(self.B, 32, dtype=torch.int32, device=device),
                      "out_probs": torch.empty(self.B, 32, dtype=torch.float32, device=device),
                      "status": torch.empty(self.B, dtype=torch.int32, device=device)} for _ in range(n_steps)]
        self.n_launch = 0
        torch.cuda.synchronize()

    def reset(self):
        pass

    def step(self, i):
        tgt, dft, drafts, u, _ = self.sets[i % 2]
        self.sv.verify_logits(tgt, dft, drafts, u, self.T, self.k, self.p, workspace=self.ws, out=self.outs[i])
        self.n_launch += 2          # the streaming pass and the per-row pass

    def launches(self):
        return self.n_launch

    def check(self, i0, n):
        em = sum(int(self.outs[i]["accepted_len"].sum().item()) + self.B for i in range(i0, i0 + n))
        ok = all(int(self.outs[i]["status"].abs().sum().item()) == 0 for i in range(i0, i0 + n))
        return ok, em

    def profile(self, n):
        import torch
        ms = []
        # one untimed step first: the host then stays ahead of the GPU, so each timed launch
        # starts as soon as the previous one ends, as in the timed loop
        self.step(0)
        for i in range(n):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            self.step(i)
            b.record()
            ms.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ms]

    def roofline(self, prof, peaks):
        avg = sum(prof) / len(prof)
        achieved = self.bytes_per_step() / (avg / 1e3) / 1e9
        # DRAM bytes (read + write) of both verify kernels from one ncu capture of this
        # workload (caches flushed per kernel): pass 1 350.09 + 5.36 MB, pass 2 4.41 MB;
        # re-take it when they change
        traffic = 350.09e6 + 5.36e6 + 4.41e6 if (self.B, self.K, self.V) == (64, 4, 151936) else None
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": "verify_kernel",
                "traffic_unit": "bytes per launch",
                "algorithmic_bytes_per_launch": self.bytes_per_step(), "avg_launch_us": avg * 1e3,
                "peak_source": peaks["source"]}

    def e2e(self, n):
        import torch
        tgt, dft, drafts, u, _ = self.sets[0]
        h_in = [x.cpu().pin_memory() for x in (tgt, dft, drafts, u)]
        d_in = [torch.empty_like(x) for x in (tgt, dft, drafts, u)]
        h_out = [torch.empty(self.B, dtype=torch.int32).pin_memory() for _ in range(2)]
        st = torch.cuda.current_stream()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        emitted = 0
        for i in range(n):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            o = self.sv.verify_logits(d_in[0], d_in[1], d_in[2], d_in[3], self.T, self.k, self.p, workspace=self.ws,
                                      out=self.outs[0])
            h_out[0].copy_(o["accepted_len"], non_blocking=True)
            h_out[1].copy_(o["next_token"], non_blocking=True)
            st.synchronize()
            emitted += int(h_out[0].sum()) + self.B
        dt = time.perf_counter() - t0
        return emitted / dt, sum(x.numel() * x.element_size() for x in h_in), 2 * self.B * 4

    def oracle_sample(self, budget_s):
        from oracle import verify as ov
        tgt, dft, drafts, u, case = self.sets[0]
        d = drafts.cpu().numpy()
        t0 = time.perf_counter()
        n_seq = emitted = 0
        while time.perf_counter() - t0 < budget_s:
            b = n_seq % self.B
            r = ov.verify(case["target"][b], case["draft"][b], d[b], case["u"][b], self.T, self.k, self.p)
            emitted += r["a"] + 1
            n_seq += 1
        dt = time.perf_counter() - t0
        return emitted / dt, (f"{n_seq} sequences of the B=64 batch (each {2 * self.K + 1} rows x {self.V}), "
                              "float64 numpy, one process")


def verify_kernel_timing(dev, peaks, n=20):
    """The standalone fused verify (B = 64, K = 4, fp32 logits of 151,936 entries) timed with
    CUDA events on its stream: two 350 MB input sets alternate (above L2), 3 warm-up calls."""
    import torch
    vl = VerifyLogitsWorkload()
    vl.setup(dev, n + 3)
    for i in range(3):
        vl.step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(n):
        vl.step(3 + i)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / n * 1e3
    gbs = vl.bytes_per_step() / (us / 1e6) / 1e9
    ok, _ = vl.check(3, n)
    out = {"us_per_call": us, "algorithmic_bytes": vl.bytes_per_step(), "achieved_gbs": gbs,
           "frac_of_measured_hbm": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0, "outputs_checked": ok}
    del vl
    torch.cuda.empty_cache()
    return out


WORKLOADS = {DenseVerifyWorkload.name: DenseVerifyWorkload, VerifyLogitsWorkload.name: VerifyLogitsWorkload,
             ServingWorkload.name: ServingWorkload, SamplingWorkload.name: SamplingWorkload}
DEFAULT_WORKLOAD = DenseVerifyWorkload.name
# DRAM bytes (read + write) of one graphed 8B verify step (see DenseVerifyWorkload.roofline),
# from an ncu capture of a 2-layer slice with --cache-control none over two steps: per layer
# (the four GEMMs, attention and combine: 394.8, 391.6, 388.2 and 387.9 MB) and the rest of
# the step (embed, lm_head with its per-tile argmax keys, the greedy merge, length update:
# 1252.0 and 1248.6 MB); in that capture the small slice's KV pages stay in L2, so the full
# model's attention reads (about 4.3 MB per layer at a context of 1.1K) are not in it.
# 0 = not captured for the current kernels.
STEP_TRAFFIC_PER_LAYER = 390.6e6
STEP_TRAFFIC_FIXED = 1250.3e6


def run_reference(args):
    """The CPU oracle as it stands, on the same workload/metric (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    from oracle import verify as ov
    wl = WORKLOADS[args.workload]()
    if isinstance(wl, VerifyLogitsWorkload):
        case = synth.verify_logits_case(wl.seed, wl.B, wl.K, wl.V)
        n_per_step = 4
        drafts = np.array([[ov.sample_token(case["draft"][b, i], case["u_draft"][b, i], wl.T, wl.k, wl.p)[0]
                            for i in range(wl.K)] for b in range(n_per_step)], dtype=np.int32)

        def step():
            em = 0
            for b in range(n_per_step):
                r = ov.verify(case["target"][b], case["draft"][b], drafts[b], case["u"][b], wl.T, wl.k, wl.p)
                em += r["a"] + 1
            return em
        sample = f"{n_per_step} of the {wl.B} sequences per step"
        unit_per_step = None
    elif isinstance(wl, ServingWorkload):
        step, sample = reference_serving_step(wl)
    elif isinstance(wl, SamplingWorkload):
        step, sample = reference_sampling_step(wl)
    else:
        step, sample = reference_dense_step(wl)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    em = 0.0
    for _ in range(args.steps):
        em += step()
    dt = time.perf_counter() - t0
    val = em / dt
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(wl.config(), sample=sample), "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reference_sampling_step(wl):
    """One bounded oracle round of the sampling workload on 1-layer slices (float64, weights
    drawn on the CPU from the same seeded generators, 4096-row vocabulary): the draft
    samples K = 4 tokens from its truncated q (context 63), the target's verify pass of the
    K + 1 tokens and the oracle's rejection-sampling rule; counted as 1/64 of a round
    (the target's 64 layers dominate), emitting (a + 1) / 64 tokens."""
    import copy
    import dataclasses
    import synth
    from oracle import model as om
    from oracle import verify as ov
    decs = []
    for shp in (wl.shape, wl.dshape):
        sub = dataclasses.replace(shp, n_layers=1, vocab=4096)
        names = [n for n in synth.weight_names(sub) if n.startswith("layers.0.")]
        w = {n: om.to_f64(synth.model_weight(shp, n, seed=0)) for n in names}
        w["embed"] = om.to_f64(synth.model_weight(sub, "embed", seed=0))
        w["final_norm"] = np.ones(shp.d_model)
        w["lm_head"] = om.to_f64(synth.model_weight(sub, "lm_head", seed=0))
        decs.append(om.Decoder(sub, w))
    tgt, dft = decs
    prompt = [int(t) for t in synth.prompt_tokens(1, 64, 4096)]
    caches = []
    for dec in decs:
        c = dec.new_cache()
        dec.forward(prompt[:-1], c, logits_rows=np.zeros(0, dtype=np.int64))
        caches.append(c)
    g = np.random.Generator(np.random.PCG64(2))
    K = wl.K

    def step():
        ct, cd = copy.deepcopy(caches[0]), copy.deepcopy(caches[1])
        tok = prompt[-1]
        drafts, qrows = [], []
        for _ in range(K):
            row = dft.forward([tok], cd)[0]
            tok, _ = ov.sample_token(row, float(g.random()), wl.T, wl.k, wl.p)
            drafts.append(tok)
            qrows.append(row)
        rows = tgt.forward([prompt[-1]] + drafts, ct)
        r = ov.verify(rows, np.array(qrows), np.array(drafts), list(g.random(K + 1)), wl.T, wl.k, wl.p)
        return (r["a"] + 1) / wl.shape.n_layers

    return step, (f"one round on 1-layer slices of the target and the draft (4096-row vocabulary, context 63): "
                  f"{K} sampled draft tokens, the target pass of {K + 1} tokens and the rejection rule; counted as "
                  f"1/{wl.shape.n_layers} of a round")


def reference_serving_step(wl):
    """One bounded oracle step of the serving workload: one sequence's verify pass (the last
    committed token and its n-gram drafts, K <= 8) through one layer of the 8B shape at a
    context of 255 tokens (float64, weights drawn on the CPU from the same seeded generator,
    a 4096-row lm_head), greedy rule on its rows; counted as 1/36 of that sequence's share
    of a verify step, emitting (a + 1) / 36 tokens."""
    import dataclasses
    import synth
    from oracle import generate as og
    from oracle import model as om
    from oracle import verify as ov
    s = wl.shape
    sub = dataclasses.replace(s, n_layers=1, vocab=4096)
    names = [n for n in synth.weight_names(sub) if n.startswith("layers.0.")]
    w = {n: om.to_f64(synth.model_weight(s, n, seed=0)) for n in names}
    w["embed"] = om.to_f64(synth.model_weight(sub, "embed", seed=0))
    w["final_norm"] = np.ones(s.d_model)
    w["lm_head"] = om.to_f64(synth.model_weight(sub, "lm_head", seed=0))
    dec = om.Decoder(sub, w)
    ctx = [int(t) for t in synth.ngram_prompt(5, 256, sub.vocab)]
    drafts = og.ngram_draft(ctx, n_draft=wl.K)
    toks = [ctx[-1]] + drafts

    import copy
    cache0 = dec.new_cache()
    dec.forward(ctx[:-1], cache0, logits_rows=np.zeros(0, dtype=np.int64))

    def step():
        cache = copy.deepcopy(cache0)
        rows = dec.forward(toks, cache)
        r = ov.verify_greedy(rows, drafts)
        return (r["a"] + 1) / s.n_layers

    return step, (f"one sequence's verify pass ({len(toks)} tokens: last + n-gram drafts) through 1 of "
                  f"{s.n_layers} layers at context 255 + a 4096-row lm_head, counted as 1/{s.n_layers} of its "
                  f"share of a step")


def reference_dense_step(wl):
    """The same oracle verify step as the CPU baseline of the 8B workload."""
    return dense_oracle_step(wl.shape, wl.K, wl.alpha)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-verify-kernel", action="store_true",
                    help="skip the standalone verify-kernel timing added to the 8B workload's line")
    ap.add_argument("--profile-steps", type=int, default=10)
    ap.add_argument("--gen", type=int, default=512, help="tokens of the recorded greedy trajectory (8B workload)")
    ap.add_argument("--layers", type=int, default=None, help="layers of the 8B shape (profiler captures only)")
    ap.add_argument("--profiler-range", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import __graft_entry__
    __graft_entry__.build()
    rank, world, local = dist_setup()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    if args.workload == DenseVerifyWorkload.name:
        wl = WORKLOADS[args.workload](n_gen=args.gen, layers=args.layers)
    elif args.workload in (ServingWorkload.name, SamplingWorkload.name):
        wl = WORKLOADS[args.workload](layers=args.layers)
    else:
        wl = WORKLOADS[args.workload]()
    n_total = args.warmup + args.steps
    # a created stream: the legacy default stream serialises programmatic dependent launches
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    wl.setup(dev, max(n_total, args.profile_steps))

    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    barrier(world)

    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        barrier(world)
        l0 = wl.launches()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if args.profiler_range:
            torch.cuda.profiler.start()
        t0.record(stream)
        for i in range(args.warmup, n_total):
            wl.step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        if args.profiler_range:
            torch.cuda.profiler.stop()
        launches = wl.launches() - l0
        barrier(world)
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ok, emitted = wl.check(args.warmup, args.steps)
    extra = {}
    if getattr(wl, "device_timed", False):
        # each step also does host work (drafting, the round's download); the value counts
        # the verify calls' own CUDA-event time, the loop's span goes beside it
        extra["round_ms_per_step"] = total_ms / args.steps
        extra.update(wl.stats(args.warmup, args.steps))
        total_ms = max_over_ranks(wl.timed_ms(args.warmup, args.steps), world)
    value = emitted * world / (total_ms / 1e3)

    if isinstance(wl, DenseVerifyWorkload):
        dec_ms = wl.decode_ms(20)
        extra["decode_ms_per_step"] = dec_ms
        extra["verify_over_decode"] = (total_ms / args.steps) / dec_ms
        # the value counts the tokens the sampled draft lengths gave; the closed-form mean of
        # the scripted drafter, (1 - a^(K+1)) / (1 - a), gives the expected rate
        per_step = (1 - wl.alpha ** (wl.K + 1)) / (1 - wl.alpha)
        extra["emitted_per_step_sampled"] = emitted / (world * args.steps)
        extra["emitted_per_step_expected"] = per_step
        extra["value_at_expected_emission"] = per_step * world / (total_ms / args.steps / 1e3)
    prof = wl.profile(args.profile_steps)
    if isinstance(wl, DenseVerifyWorkload):
        roof = wl.roofline(prof, peaks, ms_per_step=total_ms / args.steps, profile_steps=args.profile_steps)
    else:
        roof = wl.roofline(prof, peaks)
    if isinstance(prof, dict):
        # an eager pass with CUDA events around every launch (no graph, no overlap between
        # kernels): where the time goes, not the timed step
        extra["kernel_breakdown_ms_per_step_instrumented"] = {k: v["ms"] / args.profile_steps for k, v in prof.items()}
        step_bytes = sum(v["bytes"] for v in prof.values()) / args.profile_steps
        extra["step_algorithmic_bytes"] = step_bytes
        extra["step_hbm_gbs"] = step_bytes / (total_ms / args.steps / 1e3) / 1e9
        extra["step_frac_of_8tbs"] = extra["step_hbm_gbs"] / 8000.0
    if isinstance(wl, DenseVerifyWorkload) and not args.no_verify_kernel:
        extra["verify_kernel_b64_k4"] = verify_kernel_timing(dev, peaks)
    e2e_val, h2d, d2h = wl.e2e(max(5, min(args.steps, 20)))
    e2e_val = e2e_val * world
    if isinstance(wl, SamplingWorkload):
        extra.update(wl.stats(args.warmup, args.steps))
        extra["k_sweep"] = wl.k_sweep()

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": dict(wl.config(), parallelism=f"replicas x{world}"),
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "outputs_checked": ok,
    }
    line.update(extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, sample = wl.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": val, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
