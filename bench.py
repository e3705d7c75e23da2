"""Benchmark of the PuzzleKV hot path on one GB300 (or N independent replicas).

A step = one decode step of a Llama-3.1-8B-shaped attention stack (32 layers,
8 KV heads, 32 query heads, d = 128, bf16, P = 64, r_K = 16, r_V = 24, sink 4
tokens, recent 128 tokens) at a 32K-token context, batch 1: for every layer,
append the new key/value (converting the page that leaves the window, once
per 64 steps per layer) and run mixed dense/factorized decode attention.
The prompt cache is factorized once before timing (pages factorized/s).

Prints one JSON line (see --help).  ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOADS = {
    # name: (layers, kv_heads, q_heads, d, P, rk, rv, sink, recent, batch, T, rope, inner rank, outliers)
    "llama32k": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=1, T=32768, rope=5e5,
                     k=12, n_out=4,
                     desc="Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d=128, bf16, "
                          "T=32768, batch 1, P=64, rK=16, rV=24, sink 4, recent 128"),
    "incremental8": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=8, T=4096, rope=5e5,
                         k=12, n_out=4, steps=4096,
                         desc="Incremental compression during generation: Llama-3.1-8B-shaped attention, 32 layers, "
                              "8 KV / 32 query heads, d=128, bf16, batch 8, 4096-token prompts then 4096 decode steps, "
                              "P=64, rK=16, rV=24, sink 4, recent 128"),
    "batched16": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=16, T=32768, rope=5e5,
                      k=12, n_out=4, steps=32, lens=(8192, 32768, 7),
                      desc="Batched serving decode, Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, "
                           "d=128, bf16, 16 requests of U[8192, 32768] tokens (seed 7), P=64, rK=16, rV=24, sink 4, "
                           "recent 128"),
    "batched16-int4": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=16, T=32768, rope=5e5,
                           k=12, n_out=4, steps=32, lens=(8192, 32768, 7), int4=True,
                           desc="Batched serving decode, Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query "
                                "heads, d=128, bf16, 16 requests of U[8192, 32768] tokens (seed 7), P=64, rK=16, "
                                "rV=24, sink 4, recent 128, INT4 factors"),
    "llama32k-int4": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=1, T=32768, rope=5e5,
                          k=12, n_out=4, int4=True,
                          desc="Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d=128, bf16, "
                               "T=32768, batch 1, P=64, rK=16, rV=24, sink 4, recent 128, INT4 factors"),
    # the pages' own setting: P = 32, (r_K, r_V) = (16, 14), a two-page recent window
    "llama32k-p32": dict(layers=32, H=8, Hq=32, d=128, P=32, rk=16, rv=14, sink=4, W=64, B=1, T=32768, rope=5e5,
                         k=12, n_out=4,
                         desc="Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d=128, bf16, "
                              "T=32768, batch 1, P=32, rK=16, rV=14, sink 4, recent 64"),
    "llama32k-p32-int4": dict(layers=32, H=8, Hq=32, d=128, P=32, rk=16, rv=14, sink=4, W=64, B=1, T=32768,
                              rope=5e5, k=12, n_out=4, int4=True,
                              desc="Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d=128, bf16, "
                                   "T=32768, batch 1, P=32, rK=16, rV=14, sink 4, recent 64, INT4 factors"),
    # keys given before RoPE: factorized unrotated, turned at attention (theta 5e5)
    "llama32k-prerope": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=1, T=32768,
                             rope=None, rope_theta=5e5, k=12, n_out=4,
                             desc="Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d=128, bf16, "
                                  "T=32768, batch 1, P=64, rK=16, rV=24, sink 4, recent 128, keys stored before "
                                  "RoPE (theta 5e5) and turned at attention"),
    # prompt processing: per-layer dense attention (PyTorch's fused causal attention
    # as the model's stand-in) followed by that layer's page factorization
    "prefill-llama32k": dict(layers=32, H=8, Hq=32, d=128, P=64, rk=16, rv=24, sink=4, W=128, B=1, T=32768,
                             rope=5e5, k=12, n_out=4, prefill=True, steps=3,
                             desc="Prompt compression during prefill, Llama-3.1-8B-shaped attention, 32 layers, "
                                  "8 KV / 32 query heads, d=128, bf16, T=32768, P=64, rK=16, rV=24, sink 4, "
                                  "recent 128; per layer: causal GQA attention over the prompt, then the "
                                  "layer's page factorization"),
    "qwen128k": dict(layers=64, H=8, Hq=64, d=128, P=64, rk=24, rv=24, sink=4, W=128, B=1, T=131072, rope=None,
                     k=12, n_out=4,
                     desc="Qwen3-32B-shaped attention, 64 layers, 8 KV / 64 query heads, d=128, bf16, "
                          "T=131072, batch 1, P=64, rK=rV=24, sink 4, recent 128"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: 64, or the workload's own count)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--workload", default="llama32k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling runs)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = WORKLOADS[args.workload].get("steps", 64)
    return args


def measured_peak_bf16():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def factorization_roofline(wl, jobs, rotations, ms, sms, sm_mhz):
    """Rates of the prefill factorization against the two peaks that bound it.
    FLOP conventions per page job (P x d page, P x P Gram, rank r):
      Gram 2 P^2 d; projection 2 r P d; Householder reduction 2 P^3 (per
      reflection a matrix-vector product and a rank-2 update of the trailing
      block, 6 n^2 summed over n < P).  Then, for r <= P / 2 (the top-r
      eigenpairs): multisection 6 rounds x 32 Sturm counts x 3 P per
      eigenvalue; inverse iteration 3 solves x 10 P per vector; Gram-Schmidt
      3 passes x 2 r^2 P; the reflections applied to r vectors 2 P^2 r.  For
      r > P / 2: forming the reflections' product 4/3 P^3 and QL 6 P + 20 per
      plane rotation (two columns of the eigenvector matrix, and the
      recurrence).  K and V jobs are half each."""
    P, d = wl["P"], wl["d"]
    sec = ms * 1e-3
    gram = jobs * 2.0 * P * P * d
    proj, eig = 0.0, jobs * 2.0 * P ** 3 + rotations * (6.0 * P + 20.0)
    for r in (wl["rk"], wl["rv"]):
        proj += jobs / 2.0 * 2.0 * r * P * d
        if 2 * r <= P:
            eig += jobs / 2.0 * (6 * 32 * 3 * P * r + 3 * 10 * P * r + 3 * 2 * r * r * P + 2 * P * P * r)
        else:
            eig += jobs / 2.0 * (4.0 / 3.0) * P ** 3
    bf16_peak, bf16_kind = measured_peak_bf16()
    fp32_peak = sms * 128 * 2 * sm_mhz * 1e6 / 1e12  # CUDA-core fp32 FMA lanes x 2 flops
    return {"page_jobs": int(jobs), "ql_rotations_per_job": round(rotations / max(jobs, 1), 1),
            "gram_tflops": round(gram / sec / 1e12, 3),
            "gram_frac_of_bf16_peak": round(gram / sec / 1e12 / bf16_peak, 6), "bf16_peak_tflops": bf16_peak,
            "bf16_peak_source": bf16_kind,
            "eigensolve_plus_projection_tflops": round((eig + proj) / sec / 1e12, 3),
            "eigensolve_frac_of_fp32_peak": round((eig + proj) / sec / 1e12 / fp32_peak, 4),
            "fp32_peak_tflops": round(fp32_peak, 1), "fp32_peak_basis": f"{sms} SMs x 128 lanes x 2 x {sm_mhz:.0f} MHz"}


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy peak is the primary denominator)


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# the sources the bf16 decode kernel is built from (a recorded ncu traffic
# figure is reported only while they are unchanged)
DECODE_SOURCES = ("decode_impl.cuh", "decode_bf16_p64.cu", "decode_bf16_q4.cu", "decode_bf16_rope.cu", "common.cuh",
                  "layout.h", "kernels.h")


def source_hash(names):
    """Hash of the sources' code: comments and whitespace do not change a kernel."""
    import re
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "page_wise_rank_gb300", "csrc", n), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, src_hash):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel_key)
        if rec and rec.get("source_hash") == src_hash:
            return rec
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pkv_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    dist.init_process_group("nccl")
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", 0))


def barrier_max(x, world):
    """Max of x over the ranks (the slowest replica sets the job's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def alg_bytes(wl, T, esz=2):
    """Algorithmic bytes of one decode-attention launch (one layer, all KV heads):
    factors of every factorized page, valid rows of every dense page, q and out."""
    import page_wise_rank_gb300 as pkv
    kinds = pkv.classify_pages(T, wl["P"], wl["sink"], wl["W"])
    n_fac = int((kinds == pkv.PAGE_FACTORED).sum())
    n_dense_tok = T - n_fac * wl["P"]
    if wl.get("int4"):  # 4-bit codes of both factors plus fp16 scales (r_K + d for K, P + d for V)
        fac = (wl["rk"] + wl["rv"]) * (wl["P"] + wl["d"]) / 2 + 2 * ((wl["rk"] + wl["d"]) + (wl["P"] + wl["d"]))
    else:
        fac = (wl["rk"] + wl["rv"]) * (wl["P"] + wl["d"]) * esz
    per_head = n_fac * fac + n_dense_tok * 2 * wl["d"] * esz
    return wl["B"] * (wl["H"] * per_head + wl["Hq"] * wl["d"] * (esz + 4))


def gpu_arm(args, rank, world, local):
    import page_wise_rank_gb300 as pkv
    import synth
    from page_wise_rank_gb300 import build as cuda_build

    wl = dict(WORKLOADS[args.workload])
    if args.layers:
        wl["layers"] = args.layers
        wl["desc"] += f" (first {args.layers} layers only)"
    cuda_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    L, H, Hq, d, P, B, T0 = wl["layers"], wl["H"], wl["Hq"], wl["d"], wl["P"], wl["B"], wl["T"]
    n_steps_total = args.warmup + args.steps * (1 if args.no_e2e else 2) + min(args.steps, 8)
    cfg = pkv.StoreConfig(num_layers=L, num_kv_heads=H, num_q_heads=Hq, head_dim=d, page_size=P, rank_k=wl["rk"],
                          rank_v=wl["rv"], sink_tokens=wl["sink"], recent_tokens=wl["W"], max_batch=B,
                          max_tokens_per_seq=T0 + n_steps_total + P + 8, kv_dtype=torch.bfloat16,
                          factor_int4=bool(wl.get("int4")), rope_theta=float(wl.get("rope_theta", 0.0)))
    spec = synth.KVSpec(layers=L, kv_heads=H, head_dim=d, page_size=P, inner_rank=wl["k"], n_outliers=wl["n_out"],
                        rope_base=wl["rope"], dtype=torch.bfloat16)
    with torch.cuda.stream(stream):
        store = pkv.Store(cfg, device=dev, stream=stream)
        # prompt cache -> factorized store (pages factorized/s), sequence slot 0 of this replica
        K = torch.empty(L, H, T0, d, dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        synth.prefill_kv(spec, T0, seq=rank, device=dev, out=(K, V))
        kinds = pkv.classify_pages(T0, P, wl["sink"], wl["W"])
        n_fact_pages = int((kinds == pkv.PAGE_FACTORED).sum()) * L * H * 2
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        store.factorize_counters(stream)  # start from zero
        store.load_prefill(0, K, V, stream=stream)
        e1.record(stream)
        st = store.check_device_status(stream)
        prefill_ms = e0.elapsed_time(e1)
        fact_jobs, fact_rot = store.factorize_counters(stream)
        if st != 0:
            raise RuntimeError(f"prefill factorization status {st}: {pkv.last_error()}")
        # the prompt's complete pages inside the window too, once, before
        # decoding (a serving loop's call after a prompt): the store's paced
        # background conversions then carry only the pages decoding completes
        store.factorize_pages(None, stream=stream)
        store.factorize_counters(stream)
        del K, V
        torch.cuda.empty_cache()
        # per-step inputs, resident in HBM before timing
        cache = {}
        qs, ks, vs = [], [], []
        for s in range(n_steps_total):
            qs.append(torch.stack([synth.queries(B, Hq, d, step=s, layer=l, device=dev) for l in range(L)]))
            kl, vl = [], []
            for l in range(L):
                k, v = synth.decode_tokens(spec, l, [rank], [T0 + s], device=dev, cache=cache)
                kl.append(k)
                vl.append(v)
            ks.append(torch.stack(kl))
            vs.append(torch.stack(vl))
        out = torch.empty(L, B, Hq, d, dtype=torch.float32, device=dev)
        seqs = [0]
        stream.synchronize()

    launches = [0]

    def step(s, ev=None, q_src=None, k_src=None, v_src=None, out_dst=None):
        qq = qs[s] if q_src is None else q_src
        kk = ks[s] if k_src is None else k_src
        vv = vs[s] if v_src is None else v_src
        T = store_len[0]
        conv = (T + 1) % P == 0  # this step completes a page (batched factorization)
        for l in range(L):
            if ev is not None:
                ev[l][0].record(stream)
            store.decode_step(l, qq[l], kk[l], vv[l], out[l], seqs, stream=stream)
            if ev is not None:
                ev[l][1].record(stream)
        # pages completed by this step: factorize them now, in one batched launch
        # over all layers, ahead of their leaving the window
        if (T + 1) % P == 0:
            if ev is not None:
                ev[L][0].record(stream)
            store.convert_ready_pages(stream=stream)
            if ev is not None:
                ev[L][1].record(stream)
            launches[0] += 1
        else:
            store.convert_ready_pages(stream=stream)  # host bookkeeping only
        launches[0] += L
        store_len[0] = T + 1
        if out_dst is not None:
            out_dst.copy_(out, non_blocking=True)
        return conv

    store_len = [T0]
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            step(s)
        stream.synchronize()
        # ---- timed region: K steps, device-resident inputs
        evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(L + 1)]
               for _ in range(args.steps)]
        t_lens = []
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        barrier(world)
        stream.synchronize()
        launches[0] = 0
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # a GPU-side sleep ahead of the start event lets the host queue work
        # before the clock starts, so host launch latency is not timed as GPU time
        # (if enqueueing is slower than the GPU, the queue drains and it shows)
        torch.cuda._sleep(20_000_000)
        s0.record(stream)
        conv_steps = []
        step_ev = [s0]
        for i in range(args.steps):
            t_lens.append(store_len[0] + 1)
            conv_steps.append(step(args.warmup + i))
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            step_ev.append(e)
        s1.record(stream)
        stream.synchronize()
        barrier(world)
        clk = clocks.stop()
        gpu_launches = launches[0]
        ms_total = barrier_max(s0.elapsed_time(s1), world)
        st = store.check_device_status(stream)
        if st != 0:
            raise RuntimeError(f"device status {st}: {pkv.last_error()}")
        # decode-attention time per layer in the timed region: steps without a
        # batched page conversion are L back-to-back decode_step launches
        step_ms = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]
        # every timed step: a step's page conversions run on the store's internal
        # stream beside the following decode steps, which they slow a little
        dec_ms = [step_ms[i] / L for i in range(args.steps)]
        dec_bytes = [alg_bytes(wl, t_lens[i]) for i in range(args.steps)]
        # the same launches one at a time (an event pair around each call stops
        # consecutive launches from overlapping), queued behind a GPU-side sleep
        n_prof = min(args.steps, 8)
        iso_ms = []
        for i in range(n_prof):
            torch.cuda._sleep(4_000_000)
            step(args.warmup + args.steps + i, ev=evs[i])
            stream.synchronize()
            iso_ms += [evs[i][l][0].elapsed_time(evs[i][l][1]) for l in range(L)]
        # ---- e2e: same steps through the public API with pinned host buffers
        e2e = None
        if not args.no_e2e:
            # a step's q, k and v packed in one pinned buffer, moved by one copy
            nq, nk = qs[0].numel(), ks[0].numel()
            hin = torch.empty(args.steps, nq + 2 * nk, dtype=torch.bfloat16).pin_memory()
            for i in range(args.steps):
                hin[i, :nq] = qs[args.warmup + i].reshape(-1).cpu()
                hin[i, nq:nq + nk] = ks[args.warmup + i].reshape(-1).cpu()
                hin[i, nq + nk:] = vs[args.warmup + i].reshape(-1).cpu()
            hout = torch.empty(args.steps, L, B, Hq, d, dtype=torch.float32).pin_memory()
            din = torch.empty(nq + 2 * nk, dtype=torch.bfloat16, device=dev)
            dq, dk, dv = (din[:nq].view(qs[0].shape), din[nq:nq + nk].view(ks[0].shape),
                          din[nq + nk:].view(vs[0].shape))
            stream.synchronize()
            barrier(world)
            x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(20_000_000)
            x0.record(stream)
            for i in range(args.steps):
                din.copy_(hin[i], non_blocking=True)
                step(args.warmup + args.steps + n_prof + i, q_src=dq, k_src=dk, v_src=dv, out_dst=hout[i])
            x1.record(stream)
            stream.synchronize()
            e2e_ms = barrier_max(x0.elapsed_time(x1), world)
            e2e = {"value": 1000.0 * e2e_ms / args.steps, "unit": "us/step",
                   "h2d_bytes_per_step": int(din.numel() * 2),
                   "d2h_bytes_per_step": int(out.numel() * 4),
                   "copies": "made by the caller on the decode stream, as a serving loop would: one "
                             "cudaMemcpyAsync of the step's q, k and v (packed, pinned host memory) before the "
                             "step's decode_step calls through the library's C ABI, one of the outputs after"}
        # ---- one batched page conversion alone: decode steps (untimed, no
        # conversion) up to the next page boundary, then the batch that the
        # boundary makes due, timed with the caller's stream waiting for it.
        # The steps cycle through the generated tokens, so the pages they
        # complete hold distinct rows like the timed steps' pages (one token
        # repeated would give pages of rank 1, which QL deflates at once)
        j = 0
        while True:
            last = (store_len[0] + 1) % P == 0
            for l in range(L):
                store.decode_step(l, qs[j % len(qs)][l], ks[j % len(ks)][l], vs[j % len(vs)][l], out[l], seqs,
                                  stream=stream)
            store_len[0] += 1
            j += 1
            if last:
                break
        stream.synchronize()
        # the store paces its batches (a new one starts when the last has
        # finished, about one CTA per SM each): time every batch the boundary
        # makes due, one after another, and add their GPU times
        store.factorize_counters(stream)
        conv_ms, conv_jobs, conv_batches = 0.0, 0, 0
        for _ in range(64):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(1_000_000)
            c0.record(stream)
            store.convert_ready_pages(stream=stream)
            store.wait_background(stream=stream)
            c1.record(stream)
            stream.synchronize()
            jobs_now = store.factorize_counters(stream)[0]
            if jobs_now == 0:
                break
            conv_ms += c0.elapsed_time(c1)
            conv_jobs += jobs_now
            conv_batches += 1
    us_step = 1000.0 * ms_total / args.steps
    dec_us = 1000.0 * sum(dec_ms) / len(dec_ms)
    achieved = sum(dec_bytes) / (sum(dec_ms) * 1e-3) / 1e9
    peak, peak_kind = measured_peak_hbm()
    src_hash = source_hash(DECODE_SOURCES)
    traffic = recorded_traffic(f"decode_bf16:{args.workload}", src_hash)
    pages_per_s = n_fact_pages / (prefill_ms * 1e-3)
    result = {
        "metric": "mixed decode attention us/step (all layers) & % HBM roofline; pages factorized/s",
        "value": round(us_step, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded low-rank-plus-noise pages, RoPE keys)",
        "config": {"workload": wl["desc"], "global_batch": wl["B"] * world, "seq_len": wl["T"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {alg_bytes(wl, T0) * L / 1e9:.2f} GB read per step"},
        "decode_attention_us_per_layer": round(dec_us, 3),
        "decode_step_us_per_layer_isolated": round(1000.0 * statistics.mean(iso_ms), 3),
        "page_conversion": {
            "how": "batched on the store's internal stream beside the decode steps, paced: a new batch "
                   "(about one CTA per SM) when the last has finished",
            "page_boundaries_in_timed_steps": sum(conv_steps),
            "boundary_every_steps": P, "page_jobs_per_boundary": conv_jobs,
            "batches_per_boundary": conv_batches,
            "ms_alone": round(conv_ms, 4),
            "amortized_us_per_step_if_serialized": round(1000.0 * conv_ms / P, 3)},
        "pages_factorized_per_s": round(pages_per_s, 1),
        "prefill_factorization": dict({"pages": n_fact_pages, "ms": round(prefill_ms, 3)},
                                      **factorization_roofline(wl, fact_jobs, fact_rot, prefill_ms,
                                                               torch.cuda.get_device_properties(dev).multi_processor_count,
                                                               (clk or {}).get("sm_mhz") or 2070.0)),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": "decode_bf16_kernel: one decode_step launch per layer (append + attention + split merge), mean over the timed steps",
                     "traffic": (traffic["bytes_per_launch"] if traffic else None),
                     "algorithmic_bytes_per_launch": int(statistics.mean(dec_bytes))},
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_sample(wl)
    store.close()
    return result


def _oracle_sample(wl, layer_heads, nthreads):
    """Oracle factorization of every eligible page of the sampled (layer, KV head)
    pairs (timed, all host threads) and oracle decode of each pair (timed, one
    thread), then the same decodes run nthreads at a time on a thread pool (the
    oracle releases the interpreter while it computes).  Returns (pages/s,
    seconds per (layer, head) decode on one thread, (layer, head) decodes per
    second on nthreads threads, pages)."""
    import oracle
    import synth

    T, P, d = wl["T"], wl["P"], wl["d"]
    spec = synth.KVSpec(layers=1, kv_heads=wl["H"], head_dim=d, page_size=P, inner_rank=wl["k"],
                        n_outliers=wl["n_out"], rope_base=wl["rope"], dtype=torch.bfloat16)
    kinds = oracle.page_kinds(T, P, wl["sink"], wl["W"])
    fac = np.nonzero(kinds == oracle.FACTORED)[0]
    n = len(kinds)
    t_fact, n_pages, t_dec, jobs = 0.0, 0, [], []
    for (layer, h) in layer_heads:
        # layer index only selects the seed; generate that layer's cache on the host
        g = synth.KVSpec(**{**spec.__dict__, "layers": layer + 1})
        K, V = synth.prefill_kv(g, T)
        Kh, Vh = K[layer, h].double().numpy(), V[layer, h].double().numpy()
        del K, V
        Xk = np.stack([Kh[p * P:(p + 1) * P] for p in fac])
        Xv = np.stack([Vh[p * P:(p + 1) * P] for p in fac])
        t0 = time.perf_counter()
        LKf, RKf, _ = oracle.factorize_pages(Xk, wl["rk"], nthreads)
        LVf, RVf, _ = oracle.factorize_pages(Xv, wl["rv"], nthreads)
        t_fact += time.perf_counter() - t0
        n_pages += 2 * len(fac)
        LK, RK = np.zeros((n, P, wl["rk"])), np.zeros((n, wl["rk"], d))
        LV, RV = np.zeros((n, P, wl["rv"])), np.zeros((n, wl["rv"], d))
        LK[fac], RK[fac], LV[fac], RV[fac] = LKf, RKf, LVf, RVf
        G = wl["Hq"] // wl["H"]
        q = synth.queries(1, wl["Hq"], d, step=0, layer=layer)[0, h * G:(h + 1) * G].double().numpy()
        t0 = time.perf_counter()
        oracle.decode_head(q, kinds, Kh, Vh, LK, RK, LV, RV, T, P)
        t_dec.append(time.perf_counter() - t0)
        jobs.append((q, kinds, Kh, Vh, LK, RK, LV, RV))
    # all host threads: each sampled pair's decode repeated so that every thread has work
    from concurrent.futures import ThreadPoolExecutor
    calls = [jobs[i % len(jobs)] for i in range(max(nthreads, len(jobs)))]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        list(ex.map(lambda a: oracle.decode_head(*a, T, P), calls))
    par_rate = len(calls) / (time.perf_counter() - t0)
    return n_pages / t_fact, statistics.mean(t_dec), par_rate, n_pages


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the machine type."""
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                name = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        name = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return f"{name or 'unknown'} ({platform.machine()})"


def tiny_oracle_run():
    """The oracle over the whole tiny workload (1 layer, 2 KV / 8 query heads,
    d = 64, fp32, T = 1024, P = 32, r = 8, sink 4, recent 64): every eligible
    page of both heads factorized (keys and values) and one decode step of all
    query heads, on one thread.  Returns seconds."""
    import oracle
    import synth

    T, P, d, r = 1024, 32, 64, 8
    spec = synth.KVSpec(layers=1, kv_heads=2, head_dim=d, page_size=P, inner_rank=6, n_outliers=2,
                        dtype=torch.float32)
    K, V = synth.prefill_kv(spec, T)
    q = synth.queries(1, 8, d, step=0, dtype=torch.float32)[0].double().numpy()
    kinds = oracle.page_kinds(T, P, 4, 64)
    fac = np.nonzero(kinds == oracle.FACTORED)[0]
    n = len(kinds)
    t0 = time.perf_counter()
    for h in range(2):
        Kh, Vh = K[0, h].double().numpy(), V[0, h].double().numpy()
        LK, RK = np.zeros((n, P, r)), np.zeros((n, r, d))
        LV, RV = np.zeros((n, P, r)), np.zeros((n, r, d))
        LK[fac], RK[fac], _ = oracle.factorize_pages(np.stack([Kh[p * P:(p + 1) * P] for p in fac]), r, 1)
        LV[fac], RV[fac], _ = oracle.factorize_pages(np.stack([Vh[p * P:(p + 1) * P] for p in fac]), r, 1)
        oracle.decode_head(q[4 * h:4 * h + 4], kinds, Kh, Vh, LK, RK, LV, RV, T, P)
    return time.perf_counter() - t0


def cpu_baseline_sample(wl):
    nthreads = os.cpu_count() or 1
    pairs = [(0, 0), (wl["layers"] - 1, wl["H"] - 1)]
    pages_s, t_head, par_rate, n_pages = _oracle_sample(wl, pairs, nthreads)
    heads = wl["layers"] * wl["H"] * wl["B"]
    # per step: attention over every (layer, KV head), plus on average 2 H L / P page conversions
    conv_per_step = 2.0 * wl["H"] * wl["layers"] * wl["B"] / wl["P"]
    us_step = 1e6 * (heads / par_rate + conv_per_step / pages_s)
    us_step_1 = 1e6 * heads * t_head
    return {"value": round(us_step, 1), "unit": "us/step", "cores": nthreads, "kind": "oracle",
            "sample": f"oracle decode of {len(pairs)} (layer, KV head) pairs at T={wl['T']}, run "
                      f"{max(nthreads, len(pairs))} times on {nthreads} threads at once, scaled to {heads} pairs per "
                      f"step, plus {conv_per_step:.0f} page conversions per step at the oracle's factorization rate",
            "decode_us_per_step_1_core": round(us_step_1, 1),
            "decode_pairs_per_s": {"1_core": round(1.0 / t_head, 3), f"{nthreads}_cores": round(par_rate, 3)},
            "pages_factorized_per_s": round(pages_s, 1), "pages_cores": nthreads, "pages_sample": n_pages,
            "nproc": nthreads, "cpu_model": cpu_model(),
            "tiny_workload_full_oracle_s": round(tiny_oracle_run(), 4)}


def multi_seq_arm(args, rank, world, local):
    """Several sequences per decode call (batch 8 incremental generation, or
    16 ragged requests): per-step latency (mean, p50, p99, the steps that
    completed pages), the decode kernel's HBM roofline, and pages/s; pages
    are converted on the store's internal stream as they complete.
    Steps are timed in chunks, each queued behind a GPU-side sleep, so the
    per-step CUDA-event deltas are GPU time, not host enqueue time."""
    import page_wise_rank_gb300 as pkv
    import synth
    from page_wise_rank_gb300 import build as cuda_build

    wl = dict(WORKLOADS[args.workload])
    if args.layers:
        wl["layers"] = args.layers
        wl["desc"] += f" (first {args.layers} layers only)"
    cuda_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    L, H, Hq, d, P, B = wl["layers"], wl["H"], wl["Hq"], wl["d"], wl["P"], wl["B"]
    lens0 = synth.batch_lengths(B, *wl["lens"][:2], seed=wl["lens"][2]) if "lens" in wl else [wl["T"]] * B
    n_steps = args.warmup + args.steps
    cfg = pkv.StoreConfig(num_layers=L, num_kv_heads=H, num_q_heads=Hq, head_dim=d, page_size=P, rank_k=wl["rk"],
                          rank_v=wl["rv"], sink_tokens=wl["sink"], recent_tokens=wl["W"], max_batch=B,
                          max_tokens_per_seq=max(lens0) + n_steps + 8, kv_dtype=torch.bfloat16,
                          factor_int4=bool(wl.get("int4")))
    spec = synth.KVSpec(layers=L, kv_heads=H, head_dim=d, page_size=P, inner_rank=wl["k"], n_outliers=wl["n_out"],
                        rope_base=wl["rope"], dtype=torch.bfloat16)
    seqs = list(range(B))
    with torch.cuda.stream(stream):
        store = pkv.Store(cfg, device=dev, stream=stream)
        prefill_ms = 0.0
        store.factorize_counters(stream)
        for i in seqs:  # prompts: one whole-cache factorization per sequence
            K, V = synth.prefill_kv(spec, lens0[i], seq=rank * B + i, device=dev)
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            store.load_prefill(i, K, V, stream=stream)
            e1.record(stream)
            stream.synchronize()
            prefill_ms += e0.elapsed_time(e1)
            del K, V
        pre_jobs, pre_rot = store.factorize_counters(stream)
        store.factorize_pages(None, stream=stream)  # the prompts' complete window pages, once, before decoding
        store.factorize_counters(stream)
        # decode-phase inputs of every step, on the device: [L, steps, B, H, d]
        kdec = torch.empty(L, n_steps, B, H, d, dtype=torch.bfloat16, device=dev)
        vdec = torch.empty_like(kdec)
        for l in range(L):
            for i in seqs:
                k, v = synth.decode_rows(spec, l, rank * B + i, lens0[i], n_steps, device=dev)
                kdec[l, :, i] = k.transpose(0, 1)
                vdec[l, :, i] = v.transpose(0, 1)
        qs = [[synth.queries(B, Hq, d, step=s, layer=l).to(dev) for l in range(L)] for s in range(8)]
        out = torch.empty(L, B, Hq, d, dtype=torch.float32, device=dev)
        T = list(lens0)

        def step(s):
            conv = any((t + 1) % P == 0 for t in T)  # this step completes a page: batched conversion
            for l in range(L):
                store.decode_step(l, qs[s % 8][l], kdec[l, s], vdec[l, s], out[l], seqs, stream=stream)
            store.convert_ready_pages(stream=stream)
            for i in seqs:
                T[i] += 1
            return conv

        for s in range(args.warmup):
            step(s)
        stream.synchronize()
        store.factorize_counters(stream)
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        barrier(world)
        step_ms, burst, step_bytes = [], [], []
        chunk = 16
        for c0 in range(args.warmup, n_steps, chunk):
            torch.cuda._sleep(20_000_000)  # lets the host queue the chunk before the GPU reaches it
            evs = [torch.cuda.Event(enable_timing=True)]
            evs[0].record(stream)
            for s in range(c0, min(c0 + chunk, n_steps)):
                step_bytes.append(sum(alg_bytes(dict(wl, B=1), t + 1) for t in T) * L)
                burst.append(step(s))
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                evs.append(e)
            stream.synchronize()
            step_ms += [evs[i].elapsed_time(evs[i + 1]) for i in range(len(evs) - 1)]
        barrier(world)
        clk = clocks.stop()
        conv_jobs, conv_rot = store.factorize_counters(stream)
        st = store.check_device_status(stream)
        if st != 0:
            raise RuntimeError(f"device status {st}: {pkv.last_error()}")
    us = sorted(1000.0 * x for x in step_ms)
    q = lambda f: us[min(len(us) - 1, int(round(f * (len(us) - 1))))]
    burst_us = [1000.0 * step_ms[i] for i in range(len(step_ms)) if burst[i]]
    plain_us = [1000.0 * step_ms[i] for i in range(len(step_ms)) if not burst[i]]
    mean_us = barrier_max(statistics.mean(us), world)
    peak, peak_kind = measured_peak_hbm()
    achieved = sum(step_bytes) / (sum(step_ms) * 1e-3) / 1e9
    extra_burst_ms = sum(burst_us) / 1000.0 - len(burst_us) * (statistics.mean(plain_us) if plain_us else 0) / 1000.0
    return {
        "metric": "mixed decode attention us/step (all layers, conversion included) & pages factorized/s",
        "value": round(mean_us, 3), "unit": "us/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(mean_us / 1000.0, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded low-rank-plus-noise pages, RoPE keys; decode rows from the same model)",
        "config": {"workload": wl["desc"], "global_batch": B * world, "seq_len": max(lens0) + n_steps,
                   "prompt_lengths": lens0,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "chunks of 16 steps behind a GPU-side sleep; per-step CUDA events"},
        "step_latency_us": {"mean": round(statistics.mean(us), 2), "p50": round(q(0.5), 2), "p99": round(q(0.99), 2),
                            "max": round(us[-1], 2), "burst_steps": len(burst_us),
                            "burst_mean": round(statistics.mean(burst_us), 2) if burst_us else None,
                            "non_burst_mean": round(statistics.mean(plain_us), 2) if plain_us else None},
        "conversion": {"page_jobs": conv_jobs, "ql_rotations_per_job": round(conv_rot / max(conv_jobs, 1), 1),
                       "where": "store's internal low-priority stream, overlapping the decode steps",
                       "page_jobs_per_s_sustained": round(conv_jobs / (sum(step_ms) * 1e-3), 1),
                       "burst_step_excess_us": round(1000.0 * extra_burst_ms / max(len(burst_us), 1), 2)},
        "prefill_factorization": {"pages": pre_jobs, "ms": round(prefill_ms, 3),
                                  "pages_per_s": round(pre_jobs / (prefill_ms * 1e-3), 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": "decode_bf16_kernel over all layers of a step (conversion overlapped), "
                               "algorithmic bytes of every sequence",
                     "algorithmic_bytes_per_step": int(statistics.mean(step_bytes))},
        "clocks": clk,
    }


def prefill_arm(args, rank, world, local):
    """Prompt compression overlapped with prompt processing (time to first
    token).  Per layer: PyTorch's fused causal GQA attention over the whole
    prompt (the model's dense attention, not this library's work), then the
    layer's page factorization -- inline on the same stream, or in the
    background on the store's internal stream while the next layers' attention
    runs.  A step is the whole prompt; the store's state after either order is
    identical (tested)."""
    import page_wise_rank_gb300 as pkv
    import synth
    from page_wise_rank_gb300 import build as cuda_build

    wl = dict(WORKLOADS[args.workload])
    if args.layers:
        wl["layers"] = args.layers
        wl["desc"] += f" (first {args.layers} layers only)"
    cuda_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    L, H, Hq, d, P, T = wl["layers"], wl["H"], wl["Hq"], wl["d"], wl["P"], wl["T"]
    cfg = pkv.StoreConfig(num_layers=L, num_kv_heads=H, num_q_heads=Hq, head_dim=d, page_size=P, rank_k=wl["rk"],
                          rank_v=wl["rv"], sink_tokens=wl["sink"], recent_tokens=wl["W"], max_batch=1,
                          max_tokens_per_seq=T, kv_dtype=torch.bfloat16)
    spec = synth.KVSpec(layers=L, kv_heads=H, head_dim=d, page_size=P, inner_rank=wl["k"], n_outliers=wl["n_out"],
                        rope_base=wl["rope"], dtype=torch.bfloat16)
    F = torch.nn.functional
    with torch.cuda.stream(stream):
        store = pkv.Store(cfg, device=dev, stream=stream)
        K = torch.empty(L, H, T, d, dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        synth.prefill_kv(spec, T, seq=rank, device=dev, out=(K, V))
        gen = torch.Generator(device=dev).manual_seed(11)
        q = (torch.randn(1, Hq, T, d, device=dev, generator=gen) / math.sqrt(d)).to(torch.bfloat16)
        # query-head copies of the KV heads (query head h reads KV head h / G), made
        # once so that any fused attention backend serves the stand-in
        Kq = K.repeat_interleave(Hq // H, dim=1)
        Vq = V.repeat_interleave(Hq // H, dim=1)
        kinds = pkv.classify_pages(T, P, wl["sink"], wl["W"])
        jobs_per_step = int((kinds == pkv.PAGE_FACTORED).sum()) * L * H * 2

    def run(mode):
        for l in range(L):
            F.scaled_dot_product_attention(q, Kq[l:l + 1], Vq[l:l + 1], is_causal=True)
            if mode == "inline":
                store.factorize_layer(0, l, K[l], V[l], background=False, stream=stream)
            elif mode == "background":
                store.factorize_layer(0, l, K[l], V[l], background=True, stream=stream)
        if mode == "background":
            store.wait_background(stream)

    res, counters = {}, {}
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    with torch.cuda.stream(stream):
        for mode in ("attention", "inline", "background"):
            for _ in range(args.warmup):
                run(mode)
            stream.synchronize()
            store.factorize_counters(stream)
            barrier(world)
            ms = []
            for _ in range(args.steps):
                torch.cuda._sleep(20_000_000)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run(mode)
                e1.record(stream)
                stream.synchronize()
                ms.append(e0.elapsed_time(e1))
            res[mode] = barrier_max(statistics.mean(ms), world)
            counters[mode] = store.factorize_counters(stream)
        st = store.check_device_status(stream)
        if st != 0:
            raise RuntimeError(f"device status {st}: {pkv.last_error()}")
    clk = clocks.stop()
    fact_ms = res["inline"] - res["attention"]
    jobs, rot = counters["inline"]
    props = torch.cuda.get_device_properties(dev)
    fr = factorization_roofline(wl, jobs / args.steps, rot / args.steps, fact_ms, props.multi_processor_count,
                                clk.get("sm_mhz") or 2070.0)
    return {
        "metric": "prompt processing ms (dense attention of every layer + page factorization), background "
                  "factorization overlapping later layers",
        "value": round(res["background"], 3), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["background"], 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded low-rank-plus-noise pages, RoPE keys; N(0, 1/d) queries)",
        "config": {"workload": wl["desc"], "global_batch": world, "seq_len": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "CUDA events around each whole-prompt step, behind a GPU-side sleep"},
        "modes_ms": {"attention_only": round(res["attention"], 3), "factorization_inline": round(res["inline"], 3),
                     "factorization_background": round(res["background"], 3)},
        "factorization_ms_inline": round(fact_ms, 3),
        "factorization_hidden_frac": round((res["inline"] - res["background"]) / fact_ms, 4) if fact_ms > 0 else None,
        "overhead_vs_attention": {"inline": round(res["inline"] / res["attention"] - 1, 4),
                                  "background": round(res["background"] / res["attention"] - 1, 4)},
        "page_jobs_per_step": jobs_per_step,
        "roofline": {"bound": "alu", "achieved": fr["eigensolve_plus_projection_tflops"], "peak": fr["fp32_peak_tflops"],
                     "unit": "TFLOP/s", "frac": fr["eigensolve_frac_of_fp32_peak"], "traffic": None,
                     "peak_source": "derived: " + fr["fp32_peak_basis"],
                     "kernel": "factorize_kernel (prefill mode, one launch per layer), inline timing"},
        "prefill_factorization": fr,
        "clocks": clk,
        "gpu_launches": 2 * L,
    }


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    import oracle
    import synth

    T, P, d, layers, H = wl["T"], wl["P"], wl["d"], wl["layers"], wl["H"]
    nthreads = os.cpu_count() or 1
    pages_s, _, _, n_pages = _oracle_sample(wl, [(0, 0)], nthreads)
    # per step: oracle decode of one (layer, KV head) pair, scaled to all pairs
    spec = synth.KVSpec(layers=1, kv_heads=H, head_dim=d, page_size=P, inner_rank=wl["k"], n_outliers=wl["n_out"],
                        rope_base=wl["rope"], dtype=torch.bfloat16)
    K, V = synth.prefill_kv(spec, T)
    Kh, Vh = K[0, 0].double().numpy(), V[0, 0].double().numpy()
    kinds = oracle.page_kinds(T, P, wl["sink"], wl["W"])
    fac = np.nonzero(kinds == oracle.FACTORED)[0]
    n = len(kinds)
    LK, RK = np.zeros((n, P, wl["rk"])), np.zeros((n, wl["rk"], d))
    LV, RV = np.zeros((n, P, wl["rv"])), np.zeros((n, wl["rv"], d))
    a, b, _ = oracle.factorize_pages(np.stack([Kh[p * P:(p + 1) * P] for p in fac]), wl["rk"], nthreads)
    LK[fac], RK[fac] = a, b
    a, b, _ = oracle.factorize_pages(np.stack([Vh[p * P:(p + 1) * P] for p in fac]), wl["rv"], nthreads)
    LV[fac], RV[fac] = a, b
    if wl.get("int4"):  # the oracle's INT4 factors: sigma^{1/2} absorbed, quantized, dequantized exactly
        for p in fac:
            for L_, R_, per_row in ((LK, RK, False), (LV, RV, True)):
                Lt, Rt = oracle.absorb_sigma(L_[p], R_[p])
                L_[p] = oracle.dequantize_int4(*oracle.quantize_int4(Lt, per_row), per_row)
                R_[p] = oracle.dequantize_int4(*oracle.quantize_int4(Rt, False), False)
    theta = float(wl.get("rope_theta", 0.0))
    G = wl["Hq"] // H
    times = []
    for s in range(args.warmup + args.steps):
        q = synth.queries(1, wl["Hq"], d, step=s, layer=0)[0, :G].double().numpy()
        t0 = time.perf_counter()
        if theta > 0:  # keys stored before RoPE: turned at their positions
            oracle.decode_head_rope(q, kinds, Kh, Vh, LK, RK, LV, RV, T, P, theta)
        else:
            oracle.decode_head(q, kinds, Kh, Vh, LK, RK, LV, RV, T, P)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    heads = layers * H * wl["B"]
    conv_per_step = 2.0 * H * layers * wl["B"] / P
    us_step = 1e6 * (heads * statistics.mean(times) + conv_per_step / pages_s)
    sample = (f"per step: oracle decode of 1 (layer, KV head) pair at T={T} on 1 thread, scaled to {heads} pairs, "
              f"plus {conv_per_step:.0f} conversions at the oracle factorization rate ({n_pages} pages sampled "
              f"on {nthreads} threads)")
    return {"impl": "reference", "metric": "mixed decode attention us/step (all layers) & % HBM roofline; "
                                           "pages factorized/s",
            "value": round(us_step, 1), "unit": "us/step", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us_step / 1000.0, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl["desc"], "global_batch": wl["B"], "seq_len": T, "parallelism": "cpu oracle"},
            "cpu_baseline": {"value": round(us_step, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
                             "sample": sample, "pages_factorized_per_s": round(pages_s, 1),
                             "pages_cores": nthreads, "cpu_model": cpu_model()},
            "e2e": {"value": round(us_step, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        res = reference_arm(args, rank, world)
    elif WORKLOADS[args.workload].get("prefill"):
        res = prefill_arm(args, rank, world, local)
    elif WORKLOADS[args.workload].get("steps"):
        res = multi_seq_arm(args, rank, world, local)
    else:
        res = gpu_arm(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
