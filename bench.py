#!/usr/bin/env python
"""Throughput of one nanochat pretraining step (forward, loss/bpb, backward,
Muon, AdamW) on B300, printed as one JSON line.

Workload (default d20): 20 layers, d_model 1280, 10 heads x 128, 4x MLP,
vocab 65536, bf16, 32 x 2048 tokens per step drawn from a Zipf(1.1) stream
(nanochat speedrun walkthrough, lyylswood.com, section 预搜检: 32 rows of
2048 tokens per GPU, ~560M parameters).  Synthetic data, random-init
weights.  Replicas only: with --gpus N (under torchrun) every rank trains its
own replica on its own data; there is no collective on the data path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload d20|d20x8|d26|d30|eval|decode|tiny]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

  d20x8  the pages' whole optimizer step: 8 accumulated micro-batches of 32 x 2048
         (524,288 tokens), learning rates from the run's schedule (nc_lr_schedule)
  d26    depth 26 (d_model 1664, 13 heads), 2 x 16 x 2048 tokens, scheduled rates
  eval   the evaluation pass: d20 forward, loss and bits per byte over 32 x 2048
         tokens per step, no backward (its own metric: evaluation tokens/s)
  decode inference with the KV cache: prefill of 32 prompts of 1024 tokens, then one
         greedy decode step for all 32 sequences per timed step (decode tokens/s)

Kernel-level workloads (profiling harnesses, not the headline):
  --workload attn    causal attention forward+backward alone, B=32 (or --batch),
                     T=2048, H=10, D=128, bf16 Q/K/V/dO ~ N(0, 1)
  --workload optim   Muon on the 120 d20 block matrices (N(0,1) gradients) and
                     AdamW on the 65536x1280 embedding and unembedding
  --workload gemm    the d20 MLP up-projection GEMM alone: [B*2048, 1280] x
                     [5120, 1280]^T -> bf16, B = --batch
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from pretraining_step_03_b300 import shapes, synth  # noqa: E402

METRIC = "training tokens/sec and MFU (% of bf16 peak) for d20 step on 1 B300"
WORKLOADS = {
    "attn": dict(B=32, T=2048, H=10, D=128),
    "gemm": dict(B=32, T=2048, d=1280, F=5120),
    "optim": dict(depth=20, d_model=1280, n_head=10, vocab=65536),
    "d20": dict(depth=20, d_model=1280, n_head=10, vocab=65536, B=32, T=2048, n_micro=1),
    "d20x8": dict(depth=20, d_model=1280, n_head=10, vocab=65536, B=32, T=2048, n_micro=8, schedule=True),
    "d26": dict(depth=26, d_model=1664, n_head=13, vocab=65536, B=16, T=2048, n_micro=2, schedule=True),
    "d30": dict(depth=30, d_model=1920, n_head=15, vocab=65536, B=16, T=2048, n_micro=2),
    "eval": dict(depth=20, d_model=1280, n_head=10, vocab=65536, B=32, T=2048, n_micro=1),
    "decode": dict(depth=20, d_model=1280, n_head=10, vocab=65536, B=32, T=1024, n_micro=1, cache_T=2048),
    "tiny": dict(depth=2, d_model=128, n_head=2, vocab=512, B=4, T=64, n_micro=1),
}
HP = dict(muon_lr=0.02, momentum=0.95, ns_steps=5, coefs=(3.4445, -4.7750, 2.0315), lr_emb=0.2,
          lr_unemb=0.004, beta1=0.8, beta2=0.95, eps=1e-10, wd=0.0)
# The scheduled workloads take the rates above as given at width SCHED_D_REF, scale the
# AdamW ones by sqrt(SCHED_D_REF / d_model) and apply the linear warm-down multiplier over
# the last SCHED_WARMDOWN of a 20-tokens-per-parameter run (nc_lr_schedule).
SCHED_D_REF, SCHED_WARMDOWN = 1280, 0.2
EVAL_METRIC = "evaluation tokens/sec (forward, loss and bits per byte) for d20 on 1 B300"
DECODE_METRIC = "decode tokens/sec (greedy, KV cache, 32 sequences after 1024-token prompts) for d20 on 1 B300"
NOMINAL_BF16_TFLOPS = 2250.0
# Rooflines: the kernel class -> (bound, peak key).  Peaks are the measured
# copy bandwidth and library bf16 GEMM rates of this GPU pool.
ROOF = {"gemm": "tensor", "attn_fwd": "tensor", "attn_bwd": "tensor", "muon_ns": "tensor",
        "norm": "hbm", "rope": "hbm", "ce": "hbm", "embed": "hbm", "muon_elem": "hbm", "adamw": "hbm"}
# dram read+write bytes per launch site of the dominant kernel class (the step's model
# GEMMs), from an ncu capture of the current GEMM code on the step at 4 x 2048 rows (131 MB
# per site), scaled by the 8x rows of the 32 x 2048 step (the weights, 3-13 MB per site, do
# not scale, so this slightly overstates); profiles/gemm_tc2_dram_b4.md.  None when not measured.
GEMM_TRAFFIC_PER_LAUNCH = 1.05e9
# The reference arm times one bounded oracle sample per step (the driver runs
# --steps 20 --warmup 5): a 512-token row and a sixteenth of the embedding's AdamW
# keep each near ten seconds on the host.  The cpu_baseline of our own arm is one
# sample of a whole 2048-token row and the whole embedding.
REF_SAMPLE_T, REF_ADAM_ROWS = 512, 4096
CPU_SAMPLE_T = 256   # the decode baseline's prompt


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], tensor=d["bf16_tflops_sustained"], tensor_burst=d["bf16_tflops"],
                    source="measured")
    return dict(hbm=6400.0, tensor=1400.0, tensor_burst=1800.0, source="fallback")


# ---------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id):
        self.p = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(dev.index or 0)


# ---------------------------------------------------------------- oracle timing
def cpu_baseline(w, steps=1, forward_only=False, T=None, adam_rows=None):
    """The fp64 oracle as it stands, timed on a bounded sample of one step of workload w
    in a fresh process on the host cores, and scaled to the whole step.

    Per sample: the forward+backward of one 1 x T row at full widths and depth
    (forward and loss only for the evaluation pass), then the optimizer on that
    row's gradients: Muon on one square d x d matrix and on one d x 4d matrix, AdamW
    on adam_rows rows of the embedding.  The step's time is estimated as
        t_fb * (B * T_step * n_micro) / T + t_sq * 4L + t_rect * 2L + t_adam * 2V / adam_rows
    (the optimizer runs once per step).  Returns (tokens/s of the estimate, the
    per-sample estimated step times, cores, a description of the sample)."""
    Ts = min(T or w["T"], w["T"])
    ar = min(adam_rows or w["vocab"], w["vocab"])
    code = (
        "import sys, time, json, os\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import numpy as np\n"
        "import oracle\n"
        "from oracle.model import Config\n"
        "from pretraining_step_03_b300 import synth\n"
        f"w = json.loads({json.dumps(json.dumps(w))})\n"
        f"T, AR, FWD = {Ts}, {ar}, {bool(forward_only)}\n"
        "cfg = Config(w['depth'], w['d_model'], w['n_head'], w['vocab'])\n"
        "params = synth.init_params(w['depth'], w['d_model'], w['n_head'], w['vocab'], seed=0)\n"
        "tok, tgt = synth.zipf_rows(1, T, w['vocab'], seed=1)\n"
        "tb = synth.token_bytes_binomial(w['vocab'], seed=2)\n"
        "out = []\n"
        f"for _ in range({steps}):\n"
        "    t0 = time.perf_counter()\n"
        "    if FWD:\n"
        "        oracle.eval_sums(params, cfg, tok, tgt, tb)\n"
        "        out.append([time.perf_counter() - t0, 0.0, 0.0, 0.0])\n"
        "        continue\n"
        "    _, _, g = oracle.loss_and_grads(params, cfg, tok, tgt, tb)\n"
        "    t1 = time.perf_counter()\n"
        "    oracle.muon_step(params[1], g[1], np.zeros_like(g[1]), 0.02)\n"
        "    t2 = time.perf_counter()\n"
        "    oracle.muon_step(params[6], g[6], np.zeros_like(g[6]), 0.02)\n"
        "    t3 = time.perf_counter()\n"
        "    z = np.zeros((AR, w['d_model']))\n"
        "    oracle.adamw_step(params[0][:AR], g[0][:AR], z, z, 0.2, 0.8, 0.95, 1e-10, 0.0, 1)\n"
        "    out.append([t1 - t0, t2 - t1, t3 - t2, time.perf_counter() - t3])\n"
        "print(json.dumps(out))\n")
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed:\n" + r.stderr[-2000:])
    parts = json.loads(r.stdout.strip().splitlines()[-1])
    L_, n_tok = w["depth"], w["B"] * w["T"] * w.get("n_micro", 1)
    est = [fb * n_tok / Ts + (0.0 if forward_only else sq * 4 * L_ + rect * 2 * L_ + ad * 2 * w["vocab"] / ar)
           for fb, sq, rect, ad in parts]
    if forward_only:
        sample = (f"forward and loss of 1x{Ts} tokens at full widths (fp64 NumPy), scaled linearly to "
                  f"{n_tok} tokens")
    else:
        sample = (f"forward+backward of 1x{Ts} tokens at full widths, Muon on one {w['d_model']}^2 and one "
                  f"{w['d_model']}x{4 * w['d_model']} matrix, AdamW on {ar} of the {w['vocab']} embedding rows "
                  f"(fp64 NumPy); scaled to the step: fwd+bwd x {n_tok}/{Ts} tokens, Muon x {4 * L_} square "
                  f"+ {2 * L_} rectangular matrices, AdamW x {2 * w['vocab']}/{ar} rows")
        if Ts < w["T"]:
            sample += (f"; the {Ts}-token row undercounts attention, whose cost per token grows with the "
                       f"row length ({w['T']} in the step)")
    return n_tok / (sum(est) / len(est)), est, cores, sample


# ---------------------------------------------------------------- kernel workloads
def kernel_workload(args):
    import numpy as np
    import torch
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    pk = peaks()
    if args.workload == "gemm":
        M, K, N = args.batch * 2048, 1280, 5120
        g = torch.Generator(device=dev).manual_seed(0)
        A = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
        W = torch.randn(N, K, device=dev, generator=g).to(torch.bfloat16)
        C = torch.empty(M, N, device=dev, dtype=torch.bfloat16)

        def run():
            L.nc_gemm_bf16(M, N, K, 1, A.data_ptr(), K, 0, 0, W.data_ptr(), K, 0, 0, C.data_ptr(), N, 0,
                           L.NC_BF16, 1.0, 0.0, 0, 0, s)

        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        tf = 2.0 * M * N * K / ms / 1e9
        line = {"metric": "bf16 GEMM TFLOP/s (d20 MLP up-projection shape)", "value": tf, "unit": "TFLOP/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "gemm", "M": M, "N": N, "K": K},
                "frac_burst": tf / pk["tensor_burst"], "bytes_min": 2.0 * (M * K + N * K + M * N)}
        print(json.dumps(line), flush=True)
        return
    if args.workload == "attn":
        B, T, H, D = args.batch, 2048, 10, 128
        g = torch.Generator(device=dev).manual_seed(0)
        qkv = torch.randn(B * T, 3 * H * D, device=dev, generator=g).to(torch.bfloat16)
        dout = torch.randn(B * T, H * D, device=dev, generator=g).to(torch.bfloat16)
        o = torch.empty(B * T, H * D, device=dev, dtype=torch.bfloat16)
        dqkv = torch.empty_like(qkv)
        lse = torch.empty(B, H, T, device=dev, dtype=torch.float32)
        ws = torch.empty(L.nc_attention_workspace_bytes(B, T, H), device=dev, dtype=torch.uint8)
        q, k, v = (qkv.data_ptr() + i * H * D * 2 for i in range(3))
        dq, dk, dv = (dqkv.data_ptr() + i * H * D * 2 for i in range(3))

        def fwd():
            L.nc_attention_forward(q, k, v, 3 * H * D, o.data_ptr(), H * D, lse.data_ptr(), B, T, H, D,
                                   L.NC_BF16, s)

        def bwd():
            L.nc_attention_backward(q, k, v, 3 * H * D, o.data_ptr(), dout.data_ptr(), H * D,
                                    lse.data_ptr(), dq, dk, dv, 3 * H * D, ws.data_ptr(), B, T, H, D,
                                    L.NC_BF16, s)

        causal = 0.5 * T * (T + 1)
        fl_f = 4.0 * B * H * D * causal
        res = {}
        for name, fn, fl in (("fwd", fwd, fl_f), ("bwd", bwd, 2.5 * fl_f)):
            for _ in range(args.warmup):
                fwd(); fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            res[name] = {"ms": ms, "tflops": fl / ms / 1e9, "frac": fl / ms / 1e9 / pk["tensor_burst"]}
        tot_ms = res["fwd"]["ms"] + res["bwd"]["ms"]
        line = {"metric": "causal attention fwd+bwd TFLOP/s (algorithmic, causal half)",
                "value": 3.5 * fl_f / tot_ms / 1e9, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": tot_ms, "higher_is_better": True, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": "attn", "B": B, "T": T, "H": H, "D": D},
                "parts": res, "peak_tflops_burst": pk["tensor_burst"]}
    else:
        m = Model(20, 1280, 10, 65536, 0, 0, dtype="bf16", seed=0, device=dev)
        rng = np.random.default_rng(0)
        for i in range(m.n_params):
            r, c = m.shapes[i]
            m.set_grad(i, rng.standard_normal((r, c), dtype=np.float32))

        def step(i):
            m.muon_step(HP["muon_lr"], HP["momentum"], True, HP["ns_steps"], HP["coefs"])
            m.adamw_step(HP["lr_emb"], HP["lr_unemb"], HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], i + 1)

        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        L.nc_profile(m.h, 1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        kernels = {}
        for c in (7, 8, 9):
            kms, n, fl, by = L.nc_profile_read(m.h, c)
            name = L.PROF_NAMES[c]
            ach = (fl / kms / 1e9) if ROOF[name] == "tensor" else (by / kms / 1e6)
            peak = pk["tensor_burst"] if ROOF[name] == "tensor" else pk["hbm"]
            kernels[name] = {"ms": kms / args.steps, "achieved": ach,
                             "unit": "TFLOP/s" if ROOF[name] == "tensor" else "GB/s", "frac": ach / peak}
        line = {"metric": "Muon (120 d20 matrices, 5 NS steps) + AdamW (2 x 65536x1280) step time",
                "value": ms, "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms, "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "optim"}, "kernels": kernels}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main
# ---------------------------------------------------------------- evaluation pass
def profiled_pass(L, m, run, n, barrier):
    """The per-kernel-class breakdown comes from n more steps run after the timed region
    with the library's CUDA-event profiler on (its events are kept out of the timing)."""
    L.nc_profile(m.h, 1)
    for i in range(n):
        run(i)
    barrier()
    L.nc_profile(m.h, 0)
    return n


def kernel_table(L, m, steps, pk):
    kernels = {}
    for c, name in enumerate(L.PROF_NAMES):
        kms, n, fl, by = L.nc_profile_read(m.h, c)
        if n == 0:
            continue
        if ROOF[name] == "tensor":
            ach = fl / (kms * 1e-3) / 1e12
            peak, unit = pk["tensor"], "TFLOP/s"
        else:
            ach = by / (kms * 1e-3) / 1e9
            peak, unit = pk["hbm"], "GB/s"
        kernels[name] = {"ms_per_step": kms / steps, "launch_sites_per_step": n / steps,
                         "achieved": ach, "unit": unit, "peak": peak, "frac": ach / peak}
    return kernels


def eval_workload(args):
    """d20 forward + loss + bits per byte over 32 x 2048 tokens per step, no backward;
    the byte-weighted sums run across the steps as over a validation set."""
    w = WORKLOADS["eval"]
    from pretraining_step_03_b300 import replicas
    rank, world, local = replicas.rank_env()
    B, T = w["B"], w["T"]
    fpt = shapes.eval_flops_per_token(w["depth"], w["d_model"], w["vocab"], T)
    config = {"workload": "eval", "depth": w["depth"], "d_model": w["d_model"], "n_head": w["n_head"],
              "vocab": w["vocab"], "batch": B * world, "seq_len": T, "parallelism": f"replicas{world}",
              "tokens": "zipf(1.1)", "l2": "inputs larger than L2 (8.6 GB of logits per step)"}
    if args.impl == "reference":
        if rank != 0:
            return
        _, est, cores, sample = cpu_baseline(w, steps=args.warmup + args.steps, forward_only=True,
                                             T=REF_SAMPLE_T)
        t = est[args.warmup:] if len(est) > args.warmup else est
        v = B * T / (sum(t) / len(t))
        print(json.dumps({"metric": EVAL_METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
                          "steps": len(t), "warmup": args.warmup, "ms_per_step": 1000 * sum(t) / len(t),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config, "impl": "reference",
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    import numpy as np
    import torch
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    tok, tgt = synth.zipf_rows(B, T, w["vocab"], seed=replicas.data_seed(rank) + 100)
    tb_host = synth.token_bytes_binomial(w["vocab"], seed=2)
    m = Model(w["depth"], w["d_model"], w["n_head"], w["vocab"], B, T, dtype="bf16", seed=0, device=dev)
    tb = torch.from_numpy(tb_host).to(dev)
    tok_d = torch.from_numpy(tok.reshape(-1)).to(dev)
    tgt_d = torch.from_numpy(tgt.reshape(-1)).to(dev)
    sums = torch.zeros(3, dtype=torch.float64, device=dev)
    loss_d = torch.zeros(2, dtype=torch.float32, device=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        m.eval_loss(tok_d, tgt_d, tb, B, T, accumulate=int(i > 0), sums=sums, out=loss_d)
    barrier()
    stream = torch.cuda.current_stream(dev)
    clocks = Clocks(gpu_id_for(torch, dev))
    time.sleep(0.4)
    launches0 = L.nc_launch_count()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        m.eval_loss(tok_d, tgt_d, tb, B, T, accumulate=int(i > 0), sums=sums, out=loss_d)
    e1.record(stream)
    barrier()
    launches = L.nc_launch_count() - launches0
    clk = clocks.stop()
    ms = replicas.max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
    pk = peaks()
    n_prof = profiled_pass(L, m, lambda i: m.eval_loss(tok_d, tgt_d, tb, B, T, accumulate=1, sums=sums,
                                                        out=loss_d), args.steps, barrier)
    kernels = kernel_table(L, m, n_prof, pk)
    s_host = sums.cpu().numpy()
    loss = loss_d.cpu().numpy()
    g = kernels.get("gemm")
    roofline = None
    if g:
        kms, n, fl, by = L.nc_profile_read(m.h, 0)
        roofline = {"bound": "tensor", "kernel": "gemm_tc2_kernel (the forward GEMMs, CTA pairs)",
                    "achieved": g["achieved"], "peak": pk["tensor"], "unit": "TFLOP/s", "frac": g["frac"],
                    "peak_kind": f"bf16 sustained ({pk['source']})", "traffic": None,
                    "flops_per_launch": fl / n}
    # end to end: pinned host tokens/targets in, the running sums out, every step
    tok_h = torch.from_numpy(tok.reshape(-1).copy()).pin_memory()
    tgt_h = torch.from_numpy(tgt.reshape(-1).copy()).pin_memory()
    sums_h = torch.zeros(3, dtype=torch.float64).pin_memory()
    tok_s, tgt_s = torch.empty_like(tok_d), torch.empty_like(tgt_d)

    def host_step(i):
        tok_s.copy_(tok_h, non_blocking=True)
        tgt_s.copy_(tgt_h, non_blocking=True)
        m.eval_loss(tok_s, tgt_s, tb, B, T, accumulate=int(i > 0), sums=sums)
        sums_h.copy_(sums, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    host_step(0)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        host_step(i + 1)
    barrier()
    e2e_s = replicas.max_over_ranks((time.perf_counter() - t0) / args.steps, dist, dev)
    value = replicas.job_rate(world, B * T, ms * 1e-3)
    line = {
        "metric": EVAL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
        "mfu": {"nominal_2250": value / world * fpt / (NOMINAL_BF16_TFLOPS * 1e12),
                "measured_sustained": value / world * fpt / (pk["tensor"] * 1e12),
                "flop_per_token": fpt},
        "loss": float(loss[0]), "bpb": float(loss[1]),
        "bpb_over_steps": float(s_host[1] / (np.log(2.0) * s_host[2])) if s_host[2] > 0 else None,
        "device_flag": m.check_flag(), "gpu_launches": int(launches), "roofline": roofline,
        "kernels": kernels,
        "e2e": {"value": replicas.job_rate(world, B * T, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * B * T * 4, "d2h_bytes_per_step": 24, "ms_per_step": 1000 * e2e_s},
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, _, cores, sample = cpu_baseline(w, steps=1, forward_only=True)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------- inference with the KV cache
def oracle_decode_time(w):
    """The oracle's cache-free greedy step (the full forward over a 1 x 256 prompt)."""
    code = (
        "import sys, time, json\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import oracle\n"
        "from oracle.model import Config\n"
        "from oracle import generate as og\n"
        "from pretraining_step_03_b300 import synth\n"
        f"w = json.loads({json.dumps(json.dumps(w))})\n"
        f"T = {CPU_SAMPLE_T}\n"
        "cfg = Config(w['depth'], w['d_model'], w['n_head'], w['vocab'])\n"
        "params = synth.init_params(w['depth'], w['d_model'], w['n_head'], w['vocab'], seed=0)\n"
        "tok, _ = synth.zipf_rows(1, T, w['vocab'], seed=1)\n"
        "t0 = time.perf_counter()\n"
        "og.greedy(params, cfg, tok, 1)\n"
        "print(json.dumps({'T': T, 'time': time.perf_counter() - t0}))\n")
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed:\n" + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["T"], d["time"], cores


def decode_workload(args):
    w = WORKLOADS["decode"]
    from pretraining_step_03_b300 import replicas
    rank, world, local = replicas.rank_env()
    B, T0, cT = w["B"], w["T"], w["cache_T"]
    L_, d, V = w["depth"], w["d_model"], w["vocab"]
    config = {"workload": "decode", "depth": L_, "d_model": d, "n_head": w["n_head"], "vocab": V,
              "batch": B * world, "prompt_len": T0, "cache_T": cT, "parallelism": f"replicas{world}",
              "tokens": "zipf(1.1) prompts, greedy continuation",
              "l2": "inputs larger than L2 (1.1 GB of weights and 3.4+ GB of KV cache read per step)"}
    sample_line = "greedy next token after a 1x256 prompt by the cache-free definition (full fp64 forward)"
    if args.impl == "reference":
        if rank != 0:
            return
        Tc, t, cores = oracle_decode_time(w)   # one bounded sample (a d20 fp64 forward)
        times = [t]
        v = 1.0 / t
        print(json.dumps({"metric": DECODE_METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
                          "steps": len(times), "warmup": 0, "ms_per_step": 1000 / v, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": config, "impl": "reference",
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                           "sample": sample_line},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    import numpy as np
    import torch
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    # the first four steps record the two alternating buffer pairs' CUDA graphs (a step is
    # recorded on its second use); they run before the W warm-up steps, untimed
    REC = 4
    if T0 + REC + args.warmup + 3 * args.steps + 3 > cT:
        raise SystemExit("decode: prompt + steps exceed the cache")
    prompt, _ = synth.zipf_rows(B, T0, V, seed=replicas.data_seed(rank) + 200)
    m = Model(L_, d, w["n_head"], V, B, cT, dtype="bf16", seed=0, device=dev)
    cache = m.kv_cache(B, cT)
    toks = torch.zeros(1 + REC + args.warmup + 2 * args.steps + 1, B, dtype=torch.int32, device=dev)
    p_d = torch.from_numpy(prompt.reshape(-1)).to(dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # prefill (timed on its own: a second call overwrites the same cache rows)
    m.prefill(cache, p_d, B, T0, next_tok=toks[0])
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    m.prefill(cache, p_d, B, T0, next_tok=toks[0])
    e1.record(stream)
    barrier()
    prefill_ms = e0.elapsed_time(e1)
    # two fixed token buffers in turn: from the third step on every step replays a graph
    buf = [toks[0].clone(), torch.empty_like(toks[0])]

    def dstep(i):
        m.decode_step(cache, buf[i % 2], B, T0 + i, next_tok=buf[(i + 1) % 2])

    for i in range(REC + args.warmup):
        dstep(i)
    barrier()
    clocks = Clocks(gpu_id_for(torch, dev))
    time.sleep(0.4)
    launches0 = L.nc_launch_count()
    barrier()
    e0.record(stream)
    for i in range(REC + args.warmup, REC + args.warmup + args.steps):
        dstep(i)
    e1.record(stream)
    barrier()
    launches = L.nc_launch_count() - launches0
    clk = clocks.stop()
    ms = replicas.max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
    pk = peaks()
    i0 = REC + args.warmup + args.steps
    n_prof = profiled_pass(L, m, lambda i: dstep(i0 + i), args.steps, barrier)   # (direct launches)
    kernels = kernel_table(L, m, n_prof, pk)
    flag = m.check_flag()
    # algorithmic bytes of one decode step: every weight once, the cache read up to the
    # step's position (mean over the timed steps) and the new k, v written
    n_mean = T0 + REC + args.warmup + (args.steps + 1) / 2.0
    wbytes = (12 * d * d * L_ + V * d) * 2
    kvbytes = 2 * L_ * B * n_mean * d * 2 + 2 * L_ * B * d * 2
    achieved = (wbytes + kvbytes) / (ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "the decode step (weights by the swapped tcgen05 GEMMs, cache by "
                "the TMA-fed decode attention)", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "peak_kind": f"copy bandwidth ({pk['source']})",
                "traffic": None, "bytes_per_step": wbytes + kvbytes}
    # end to end: this step's tokens from pinned host memory in, the next tokens out
    tok_h = torch.from_numpy(buf[0].cpu().numpy().copy()).pin_memory()
    nxt_h = torch.zeros(B, dtype=torch.int32).pin_memory()
    t_in = torch.empty(B, dtype=torch.int32, device=dev)
    t_out = torch.empty(B, dtype=torch.int32, device=dev)

    def host_step(pos):
        t_in.copy_(tok_h, non_blocking=True)
        m.decode_step(cache, t_in, B, pos, next_tok=t_out)
        nxt_h.copy_(t_out, non_blocking=True)
        stream.synchronize()
        tok_h.copy_(nxt_h)

    base = T0 + REC + args.warmup + 2 * args.steps    # (every position up to here has been written)
    host_step(base)
    host_step(base)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        host_step(base + 1 + i)
    barrier()
    e2e_s = replicas.max_over_ranks((time.perf_counter() - t0) / args.steps, dist, dev)
    value = replicas.job_rate(world, B, ms * 1e-3)
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
        "prefill": {"ms": prefill_ms, "tokens_per_s": B * T0 / (prefill_ms * 1e-3)},
        "graph_recording_steps": REC,
        "device_flag": flag, "gpu_launches": int(launches), "roofline": roofline, "kernels": kernels,
        "e2e": {"value": replicas.job_rate(world, B, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": B * 4,
                "d2h_bytes_per_step": B * 4, "ms_per_step": 1000 * e2e_s},
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Tc, t, cores = oracle_decode_time(w)
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample_line}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="d20", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="batch: of the attn / gemm workloads (default 32), or the micro-batch rows of a "
                         "training workload (a smaller case than the named configuration, for profiling)")
    args = ap.parse_args()
    if args.workload in ("attn", "optim", "gemm"):
        if args.batch is None:
            args.batch = 32
        return kernel_workload(args)
    if args.workload == "eval":
        return eval_workload(args)
    if args.workload == "decode":
        return decode_workload(args)
    w = dict(WORKLOADS[args.workload])
    if args.batch is not None:
        w["B"] = args.batch
    from pretraining_step_03_b300 import replicas
    rank, world, local = replicas.rank_env()
    tokens_per_step = w["B"] * w["T"] * w["n_micro"]
    fpt = shapes.flops_per_token(w["depth"], w["d_model"], w["vocab"], w["T"])
    fpt_causal = shapes.flops_per_token(w["depth"], w["d_model"], w["vocab"], w["T"], causal=True)
    config = {"workload": args.workload, "depth": w["depth"], "d_model": w["d_model"],
              "n_head": w["n_head"], "vocab": w["vocab"], "global_batch": w["B"] * w["n_micro"] * world,
              "micro_batch": w["B"], "grad_accum": w["n_micro"], "seq_len": w["T"],
              "parallelism": f"replicas{world}", "tokens": "zipf(1.1)",
              "l2": "inputs larger than L2 (47+ GB activation stash per step)"}
    if w.get("schedule"):
        config["lr_schedule"] = {"run_steps": shapes.chinchilla_steps(w["depth"], w["d_model"], w["n_head"],
                                                                      w["vocab"], tokens_per_step),
                                 "warmdown_frac": SCHED_WARMDOWN, "d_ref": SCHED_D_REF}

    if args.impl == "reference":
        if rank != 0:
            return
        _, est, cores, sample = cpu_baseline(w, steps=args.warmup + args.steps, T=REF_SAMPLE_T,
                                             adam_rows=REF_ADAM_ROWS)
        t = est[args.warmup:] if len(est) > args.warmup else est
        v = tokens_per_step / (sum(t) / len(t))
        line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world, "steps": len(t),
                "warmup": args.warmup, "ms_per_step": 1000 * sum(t) / len(t), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config, "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import numpy as np
    import torch
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ------------------------------------------------ inputs (seeded per rank)
    nm, B, T = w["n_micro"], w["B"], w["T"]
    tok, tgt = synth.zipf_rows(nm * B, T, w["vocab"], seed=replicas.data_seed(rank))
    tb_host = synth.token_bytes_binomial(w["vocab"], seed=2)
    m = Model(w["depth"], w["d_model"], w["n_head"], w["vocab"], B, T, dtype="bf16", seed=0, device=dev)
    tb = torch.from_numpy(tb_host).to(dev)
    tok_d = torch.from_numpy(tok.reshape(nm, B * T)).to(dev)
    tgt_d = torch.from_numpy(tgt.reshape(nm, B * T)).to(dev)
    loss_d = torch.zeros(nm, 2, dtype=torch.float32, device=dev)

    n_run = shapes.chinchilla_steps(w["depth"], w["d_model"], w["n_head"], w["vocab"], tokens_per_step)

    def rates(i):
        if not w.get("schedule"):
            return HP["muon_lr"], HP["lr_emb"], HP["lr_unemb"]
        return L.nc_lr_schedule(i % n_run, n_run, SCHED_WARMDOWN, w["d_model"], SCHED_D_REF,
                                (HP["muon_lr"], HP["lr_emb"], HP["lr_unemb"]))

    def step(i):
        lr_m, lr_e, lr_u = rates(i)
        for j in range(nm):
            m.forward_backward(tok_d[j], tgt_d[j], tb, B, T, accumulate=int(j > 0), grad_scale=1.0 / nm,
                               out=loss_d[j])
        m.muon_step(lr_m, HP["momentum"], True, HP["ns_steps"], HP["coefs"])
        m.adamw_step(lr_e, lr_u, HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], i + 1)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        step(i)
    barrier()
    # ------------------------------------------------ device-timed region
    stream = torch.cuda.current_stream(dev)
    clocks = Clocks(gpu_id_for(torch, dev))
    time.sleep(0.4)
    launches0 = L.nc_launch_count()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record(stream)
    barrier()
    launches = L.nc_launch_count() - launches0
    clk = clocks.stop()
    ms = replicas.max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
    loss = loss_d.cpu().numpy().mean(axis=0)
    flag = m.check_flag()
    pk = peaks()
    n_prof = profiled_pass(L, m, lambda i: step(args.warmup + args.steps + i), min(args.steps, 2), barrier)
    kernels = kernel_table(L, m, n_prof, pk)
    g = kernels.get("gemm")
    roofline = None
    if g:
        kms, n, fl, by = L.nc_profile_read(m.h, 0)
        roofline = {"bound": "tensor", "kernel": "gemm_tc2_kernel (the step's GEMMs, CTA pairs)", "achieved": g["achieved"],
                    "peak": pk["tensor"], "unit": "TFLOP/s", "frac": g["frac"],
                    "peak_kind": f"bf16 sustained ({pk['source']})",
                    "traffic": GEMM_TRAFFIC_PER_LAUNCH,
                    "flops_per_launch": fl / n}

    # ------------------------------------------------ end to end through the C ABI (host buffers)
    e2e = None
    h2d = 2 * nm * B * T * 4
    tok_h = torch.from_numpy(tok.reshape(-1).copy()).pin_memory()
    tgt_h = torch.from_numpy(tgt.reshape(-1).copy()).pin_memory()

    def host_step(i):
        lr_m, lr_e, lr_u = rates(i)
        return m.train_step(tok_h, tgt_h, tb, B, T, nm, lr_m, lr_e, lr_u, i,
                            HP["momentum"], HP["ns_steps"], HP["coefs"], HP["beta1"], HP["beta2"], HP["eps"],
                            HP["wd"])

    host_step(1000)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        host_step(1001 + i)
    barrier()
    e2e_s = replicas.max_over_ranks((time.perf_counter() - t0) / args.steps, dist, dev)
    e2e = {"value": replicas.job_rate(world, tokens_per_step, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": 8, "ms_per_step": 1000 * e2e_s}

    value = replicas.job_rate(world, tokens_per_step, ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "mfu": {"nominal_2250": value / world * fpt / (NOMINAL_BF16_TFLOPS * 1e12),
                "measured_burst": value / world * fpt / (pk["tensor_burst"] * 1e12),
                "measured_sustained": value / world * fpt / (pk["tensor"] * 1e12),
                "causal_honest_nominal": value / world * fpt_causal / (NOMINAL_BF16_TFLOPS * 1e12),
                "flop_per_token": fpt},
        "loss": float(loss[0]), "bpb": float(loss[1]), "device_flag": flag,
        "gpu_launches": int(launches),
        "roofline": roofline,
        "kernels": kernels,
        "e2e": e2e,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, _, cores, sample = cpu_baseline(w, steps=1)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
