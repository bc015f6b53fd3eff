"""Benchmark of the speculative-decoding verify step on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  Workloads:
  verify-logits-b64-k4 : the fused verify kernel alone on fp32 logits, B=64 sequences,
                         K=4 drafts, vocab 151936, temperature 1.0, top-k 20, top-p 0.95;
                         two input sets of 700 MB alternate, so no step reads L2-resident
                         data.
The metric is emitted tokens/s (accepted drafts + the correction/bonus token of every
sequence, per second of verify steps); ms_per_step is the verify-step latency and
`roofline` the achieved HBM bandwidth of the dominant kernel.
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


# ---- clocks -------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index

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
        self.lines = []
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
        for l in getattr(self, "lines", []):
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

def dist_setup(n_gpus):
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
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- workload: standalone verify on logits ----------------------------------------------

class VerifyLogitsWorkload:
    name = "verify-logits-b64-k4"

    def __init__(self, B=64, K=4, V=VOCAB, T=1.0, top_k=20, top_p=0.95, seed=3):
        self.B, self.K, self.V, self.T, self.k, self.p, self.seed = B, K, V, T, top_k, top_p, seed

    def config(self):
        return {"workload": self.name, "B": self.B, "K": self.K, "vocab": self.V, "temperature": self.T,
                "top_k": self.k, "top_p": self.p, "logits": "fp32 N(0,3^2) + shared Gumbel-perturbed spike",
                "l2": "inputs larger than L2 (two 350 MB sets alternate)"}

    def bytes_per_step(self):
        return self.B * (2 * self.K + 1) * self.V * 4

    def setup(self, device):
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
                      "status": torch.empty(self.B, dtype=torch.int32, device=device)} for _ in range(2)]
        torch.cuda.synchronize()

    def step(self, i):
        tgt, dft, drafts, u, _ = self.sets[i % 2]
        return self.sv.verify_logits(tgt, dft, drafts, u, self.T, self.k, self.p, workspace=self.ws,
                                     out=self.outs[i % 2])

    def emitted(self, i):
        return int((self.outs[i % 2]["accepted_len"].sum() + self.B).item())

    kernels_per_step = 1

    # end-to-end through the C ABI with host buffers
    def setup_e2e(self):
        import torch
        tgt, dft, drafts, u, _ = self.sets[0]
        self.h_in = [x.cpu().pin_memory() for x in (tgt, dft, drafts, u)]
        self.d_in = [torch.empty_like(x) for x in (tgt, dft, drafts, u)]
        self.h_out = [torch.empty(self.B, dtype=torch.int32).pin_memory() for _ in range(2)]
        return sum(x.numel() * x.element_size() for x in self.h_in), 2 * self.B * 4

    def step_e2e(self, i):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        o = self.sv.verify_logits(self.d_in[0], self.d_in[1], self.d_in[2], self.d_in[3], self.T, self.k, self.p,
                                  workspace=self.ws, out=self.outs[0])
        self.h_out[0].copy_(o["accepted_len"], non_blocking=True)
        self.h_out[1].copy_(o["next_token"], non_blocking=True)

    def emitted_e2e(self):
        return int(self.h_out[0].sum().item()) + self.B

    # CPU oracle on a bounded sample of the same workload
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
        return emitted / dt, f"{n_seq} sequences of the B=64 batch (each {2 * self.K + 1} rows x {self.V}), float64 numpy, one process"


WORKLOADS = {VerifyLogitsWorkload.name: VerifyLogitsWorkload}
DEFAULT_WORKLOAD = VerifyLogitsWorkload.name


def run_reference(args):
    """The CPU oracle as it stands, on the same workload/metric (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    wl = WORKLOADS[args.workload]()
    # inputs of the same workload; drafts are drawn on the CPU with the oracle's sampler
    import synth
    from oracle import verify as ov
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

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    em = 0
    for _ in range(args.steps):
        em += step()
    dt = time.perf_counter() - t0
    val = em / dt
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(wl.config(), sample=f"{n_per_step} of the {wl.B} sequences per step"),
            "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n_per_step} sequences per step x {args.steps} steps"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import __graft_entry__
    __graft_entry__.build()
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    wl = WORKLOADS[args.workload]()
    wl.setup(dev)
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    barrier(world)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    emitted = 0
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        barrier(world)
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            wl.step(i)
            ends[i].record(stream)
        t_all1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    for i in range(args.steps):
        emitted += wl.emitted(i)
    total_ms = t_all0.elapsed_time(t_all1)
    total_ms = max_over_ranks(total_ms, world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    avg_launch_ms = sum(step_ms) / len(step_ms)
    value = emitted * world / (total_ms / 1e3)

    # end-to-end: host buffers, copies inside the timed region
    h2d, d2h = wl.setup_e2e()
    for i in range(2):
        wl.step_e2e(i)
    torch.cuda.synchronize()
    e2e_steps = max(5, args.steps // 5)
    barrier(world)
    t0 = time.perf_counter()
    em_e2e = 0
    for i in range(e2e_steps):
        wl.step_e2e(i)
        torch.cuda.current_stream().synchronize()
        em_e2e += wl.emitted_e2e()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_val = em_e2e * world / e2e_s

    algo_bytes = wl.bytes_per_step()
    achieved = algo_bytes / (avg_launch_ms / 1e3) / 1e9
    traffic = getattr(wl, "dram_traffic_per_launch", None)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(wl.config(), parallelism=f"replicas x{world}"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "verify_kernel", "algorithmic_bytes_per_launch": algo_bytes,
                     "peak_source": peaks["source"]},
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "gpu_launches": wl.kernels_per_step * args.steps,
        "clocks": clk.summary(),
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, sample = wl.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
