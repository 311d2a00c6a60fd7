#!/usr/bin/env python3
"""Throughput of the GGUF-quantized Llama-style decoder forward pass on GB300.

One step = the whole workload of one synthetic config: prefill of the prompt in
512-token chunks (logits of the last chunk only), then greedy decode steps fed
from the device argmax.  Default: the Llama-3-8B-shaped Q4_0 model with a
4096-token prompt (8 chunks) and 256 decode steps over an fp16 KV cache.

Headline `value`: decode tokens/s (aggregate over ranks).  Also reported:
prefill tokens/s, decode HBM GB/s against the measured copy bandwidth
(algorithmic bytes = quantized weights + LM head + embedding row + norms +
K/V read for slots 0..pos, per token), the prefill GEMM rate, the oracle on
the host cores (cpu_baseline) and an end-to-end run through the host API.

Multi-GPU: the path does not shard at batch 1; N ranks run N independent
replicas (no collective on the data path), `scaling` = "weak".
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one gate/up GEMV launch, Q4_0 28672 x 4096, from one
# ncu capture of the kernel built from these sources (identified by their hash); reported only while they match.
GEMV_SOURCES = ["qgemv_impl.cuh", "qgemv_q4_0.cu", "gemv_common.cuh", "tma.cuh", "common.cuh"]
GEMV_TRAFFIC = {"sources_sha256_16": "ef90df1d8ee57293", "wtype": "q4_0", "N": 28672, "K": 4096, "bytes": 66182144}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured", p
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback", {}


def decode_bytes_per_token(cfg, pos):
    """Algorithmic HBM bytes of one decode step at position pos."""
    bpe = synth.BLOCK_BYTES[cfg.wtype] / synth.BLOCK_ELEMS[cfg.wtype]  # GGUF bytes per weight
    hbpe = synth.BLOCK_BYTES[cfg.head_wtype] / synth.BLOCK_ELEMS[cfg.head_wtype]
    E, QD, KVD, F, V, L = (cfg.n_embd, cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.n_ff,
                           cfg.n_vocab, cfg.n_layers)
    layer_w = (E * (QD + 2 * KVD) + QD * E + 2 * F * E + F * E) * bpe + 2 * E * 4
    head = V * E * hbpe + E * 4 + E * bpe  # LM head + final norm + one embedding row
    n = pos + 1
    if cfg.kv_dtype in ("q8_0", "q4_0"):  # retired slots from the quantized store, the window from fp16
        W = min(cfg.kv_window, n)
        kv = 2 * L * KVD * ((n - W) * synth.BLOCK_BYTES[cfg.kv_dtype] / 32 + W * 2)
    else:
        kv = 2 * L * KVD * n * (2 if cfg.kv_dtype == "f16" else 4)
    return L * layer_w + head + kv


def prefill_flops(cfg, n_tokens, chunk):
    """Algorithmic flops of prefilling n_tokens from position 0 (GEMMs + causal attention + one LM head)."""
    E, QD, KVD, F, V, L = (cfg.n_embd, cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.n_ff,
                           cfg.n_vocab, cfg.n_layers)
    params = E * (QD + 2 * KVD) + QD * E + 3 * F * E
    gemm = 2.0 * L * params * n_tokens
    attn = 4.0 * cfg.n_heads * cfg.head_dim * L * (n_tokens * (n_tokens + 1) / 2)
    return gemm + attn + 2.0 * V * E, gemm


def gemm_flops(cfg, n_tokens):
    E, QD, KVD, F, L = (cfg.n_embd, cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.n_ff,
                        cfg.n_layers)
    return 2.0 * L * (E * (QD + 2 * KVD) + QD * E + 3 * F * E) * n_tokens


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.p = None
        self.path = None

    def start(self):
        # raw samples in a temporary file (the summary goes into the JSON line); AF_CLOCKS_DIR keeps them
        out_dir = os.environ.get("AF_CLOCKS_DIR") or tempfile.gettempdir()
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if _cuda_ok() else "gloo")
    return world, rank, local


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if _cuda_ok() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle on the host cores

def oracle_sample(hm, cfg, n_decode, threads):
    """Time the oracle: a 4-token prefill then n_decode decode steps.  Returns (decode tok/s, seconds)."""
    import oracle
    om = oracle.Model.from_host(hm, kv_slots=4 + n_decode + 1)
    prompt = hm.prompt(4)
    logits, _ = om.forward(prompt, 0, nthreads=threads)
    tok = oracle.argmax(logits)
    t0 = time.perf_counter()
    for i in range(n_decode):
        logits, _ = om.forward([tok], 4 + i, nthreads=threads)
        tok = oracle.argmax(logits)
    dt = time.perf_counter() - t0
    return n_decode / dt, dt


def oracle_timing(hm, cfg, threads, n_prefill, n_decode):
    """The oracle on `threads` host threads: an n_prefill-token prefill chunk at position 0, then n_decode decode
    steps.  Returns a cpu-baseline record with both rates."""
    import oracle
    om = oracle.Model.from_host(hm, kv_slots=n_prefill + n_decode + 1)
    prompt = hm.prompt(n_prefill)
    t0 = time.perf_counter()
    logits, _ = om.forward(prompt, 0, nthreads=threads)
    t1 = time.perf_counter()
    tok = oracle.argmax(logits)
    for i in range(n_decode):
        logits, _ = om.forward([tok], n_prefill + i, nthreads=threads)
        tok = oracle.argmax(logits)
    t2 = time.perf_counter()
    return {"threads": threads, "prefill_tok_s": n_prefill / (t1 - t0), "decode_tok_s": n_decode / (t2 - t1),
            "sample": f"{n_prefill}-token prefill chunk then {n_decode} decode steps ({t2 - t0:.1f} s, fp64)"}


def oracle_baselines(hm, cfg):
    """Per-config CPU baseline: all host threads on a 4-token chunk + 2 decode steps; one thread as well where the
    model is small enough for that to take seconds (the full 64-token chunk would take minutes per config)."""
    T = os.cpu_count() or 1
    out = {"threaded": oracle_timing(hm, cfg, T, 4, 2)}
    if decode_bytes_per_token(cfg, 0) < 1.5e9:  # up to ~1.5 G weights: a few seconds single-threaded
        out["single_thread"] = oracle_timing(hm, cfg, 1, 2, 1)
    return out


def run_reference(args, cfg, world, rank):
    """The reference arm: the CPU oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    hm = synth.HostModel(cfg, synth.seed_of(args.config))
    n_dec = args.ref_decode
    for _ in range(args.warmup):
        oracle_sample(hm, cfg, 1, threads)
    total_t, total_tok = 0.0, 0
    for _ in range(args.steps):
        _, dt = oracle_sample(hm, cfg, n_dec, threads)
        total_t += dt
        total_tok += n_dec
    v = total_tok / total_t
    sample = f"{n_dec} oracle decode steps after a 4-token prefill per step, fp64, {threads} threads"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_obj(cfg, args),
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle", "cpu": cpu_name(),
                             "sample": sample},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


METRIC = "decode tok/s + HBM GB/s frac of peak (8B-shape Q4_0); prefill tok/s"


def config_obj(cfg, args):
    return {"workload": f"{cfg.name}: {args.prompt}-token prompt in {args.chunk}-token chunks + {args.decode} "
                        f"greedy decode steps, KV {cfg.kv_dtype} max_ctx {cfg.max_ctx}",
            "layers": cfg.n_layers, "n_embd": cfg.n_embd, "heads": f"{cfg.n_heads}/{cfg.n_kv_heads}x{cfg.head_dim}",
            "n_ff": cfg.n_ff, "vocab": cfg.n_vocab, "weights": cfg.wtype, "seed": synth.seed_of(args.config),
            "l2": "inputs larger than L2 (weights %.2f GB streamed per decode step)"
                  % (decode_bytes_per_token(cfg, 0) / 1e9), "parallelism": "replicas"}


# ---------------------------------------------------------------- our arm

def run_ours(args, cfg, world, rank, local):
    import torch

    import gguf_quantized_transformer_gb300 as af
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, bf16_sust, peak_src, _ = peaks()

    t0 = time.time()
    hm = synth.HostModel(cfg, synth.seed_of(args.config))
    gen_s = time.time() - t0
    layers = [torch.from_numpy(b).to(dev) for b in hm.layers]
    emb = torch.from_numpy(hm.token_embd).to(dev)
    onorm = torch.from_numpy(hm.output_norm).to(dev)
    out = torch.from_numpy(hm.output).to(dev)
    m = af.Model(cfg, layers, emb, onorm, out, max_chunk=args.chunk)
    torch.cuda.synchronize()
    del layers, emb, onorm, out
    torch.cuda.empty_cache()
    stream = torch.cuda.ExternalStream(af.af_model_stream(m.h))
    prompt = hm.prompt(args.prompt)
    prompt_dev = torch.from_numpy(prompt).to(dev)
    logits = torch.empty(cfg.n_vocab, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    P, ND, C = args.prompt, args.decode, args.chunk

    def one_step(ev):
        ev[0].record(stream)
        for p in range(0, P, C):
            n = min(C, P - p)
            last = p + n >= P
            af.af_prefill_dev(m.h, prompt_dev[p:p + n], n, p, logits if last else None)
        ev[1].record(stream)
        for i in range(ND):
            af.af_decode_step(m.h, -1, P + i, logits)
        ev[2].record(stream)

    for _ in range(args.warmup):
        one_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for k in range(args.steps):
        one_step(evs[k])
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    barrier(world)
    clk = clocks.stop()
    pre_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(args.steps)]
    dec_ms = [evs[k][1].elapsed_time(evs[k][2]) for k in range(args.steps)]
    step_ms = max_over_ranks(world, float(np.mean([a + b for a, b in zip(pre_ms, dec_ms)])))
    pre_s = max_over_ranks(world, float(np.sum(pre_ms)) / 1000)
    dec_s = max_over_ranks(world, float(np.sum(dec_ms)) / 1000)
    decode_tps = world * ND * args.steps / dec_s
    prefill_tps = world * P * args.steps / pre_s

    # decode roofline: algorithmic bytes of the timed decode steps / their time (per replica)
    dec_bytes = sum(decode_bytes_per_token(cfg, P + i) for i in range(ND))
    dec_gbs = dec_bytes * args.steps / (dec_s) / 1e9
    pf_total, pf_gemm = prefill_flops(cfg, P, C)
    pf_tflops = pf_total * args.steps / pre_s / 1e12

    # per-kernel: the decode GEMV alone, at this model's largest per-layer matrix (gate|up), CUDA events
    qg = qgemv_roofline(af, cfg, dev, hbm_peak)

    # the sampler chain over this vocabulary (typical settings), CUDA events
    samp_us = sampler_time(af, cfg, dev)

    # end to end through the host API: host token ids in, greedy token ids out, one sync per decode step
    e2e = e2e_run(af, m, prompt, cfg, args)

    # decode with the sampler chain between steps, all on the device (no logits read back)
    sampled_tps = sampled_decode(af, m, prompt_dev, cfg, args, stream)
    m.close()
    del m
    torch.cuda.empty_cache()

    # the same workload on the 8B shape in the Q4_K_M mix (Q4_K layers, Q6_K LM head): a secondary line
    tc_peak = bf16_sust or bf16_peak
    kq = None if args.no_kquant else kquant_run(af, args, dev, hbm_peak, tc_peak)
    others = config_runs(af, args, dev, hbm_peak, tc_peak)

    launches_per_step = (P + C - 1) // C * (1 + 7 * cfg.n_layers) + 3 + ND * (3 + 5 * cfg.n_layers + 1)

    line = {
        "metric": METRIC, "value": decode_tps, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (weights q4_0/q8_0 decoded exactly; fp32 accumulate)",
        "data": "synthetic (seeded random-init weights and prompt)", "config": config_obj(cfg, args),
        "prefill_tok_s": prefill_tps, "decode_tok_s": decode_tps,
        "decode_hbm_gbs": dec_gbs, "decode_hbm_frac": dec_gbs / hbm_peak,
        "prefill_tflops": pf_tflops,
        # the prefill is seconds of back-to-back GEMMs: the sustained dense bf16 figure is its denominator (the
        # same rate as fp16).  Each product runs as three MMAs (hi/lo split), so the tensor pipe does 3x this work.
        "prefill_roofline": {"bound": "tensor", "achieved": pf_tflops, "peak": bf16_sust or bf16_peak,
                             "unit": "TFLOP/s", "frac": pf_tflops / (bf16_sust or bf16_peak),
                             "pipe_work_factor": 3, "kind": "algorithmic flops (GEMMs + causal attention) / prefill time",
                             "peak_source": peak_src + (" sustained" if bf16_sust else " burst")},
        "sampler_us": samp_us,
        "decode_sampled_tok_s": sampled_tps,
        "q4_k_m": kq,
        "configs": others,
        "roofline": dict(qg, peak_source=peak_src),
        "decode_step_roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
                                 "frac": dec_gbs / hbm_peak, "traffic": None,
                                 "kernel": "decode step (GEMVs + attention + LM head; per-token algorithmic bytes = "
                                           "quantized weights + KV read)", "peak_source": peak_src},
        "cpu_baseline": None,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed": wall, "gen_s": gen_s,
    }
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        v, dt = oracle_sample(hm, cfg, args.ref_decode, threads)
        line["cpu_baseline"] = {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle", "cpu": cpu_name(),
                                "sample": f"{args.ref_decode} decode steps after a 4-token prefill "
                                          f"({dt:.1f} s, fp64, {threads} threads)",
                                "per_config": {cfg.name: oracle_baselines(hm, cfg),
                                               **{k: v.get("cpu_baseline") for k, v in others.items()
                                                  if isinstance(v, dict)}}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def sampled_decode(af, m, prompt_dev, cfg, args, stream):
    """The workload's decode phase with af_model_sample (penalty 1.1 on the prompt's last 64 ids, temperature 0.8,
    top-p 0.95, seeded uniforms) between the steps; each step reads the drawn token from the device."""
    import torch
    P, ND, C = args.prompt, args.decode, args.chunk
    if P + 1 + ND > cfg.max_ctx or P < 64:
        return None
    recent = prompt_dev[-64:].contiguous()
    us = np.random.default_rng(1).random(ND).astype(np.float32) * 0.999
    for p in range(0, P, C):
        n = min(C, P - p)
        af.af_prefill_dev(m.h, prompt_dev[p:p + n], n, p, None)
    af.af_model_sample(m.h, None, recent, 64, 1.1, 0.8, 0.95, float(us[0]))
    af.af_decode_step(m.h, -1, P, None)  # untimed: the step's graph for the model's own logits buffer is built here
    af.af_model_sample(m.h, None, recent, 64, 1.1, 0.8, 0.95, float(us[0]))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(ND):
        af.af_decode_step(m.h, -1, P + 1 + i, None)
        af.af_model_sample(m.h, None, recent, 64, 1.1, 0.8, 0.95, float(us[i]))
    b.record(stream)
    b.synchronize()
    return ND / (a.elapsed_time(b) / 1000)


def cpu_name():
    """The host CPU, as far as /proc/cpuinfo names it (x86: model name; Arm: implementer and part)."""
    import platform
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    name = fields.get("model name") or " ".join(
        f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields)
    return f"{platform.machine()} {name}".strip()


def workload_run(af, cfg, seed, P, ND, C, dev, hbm_peak, tc_peak, steps=2, warmup=1, cpu=False):
    """Prefill of a P-token prompt in C-token chunks + ND greedy decode steps of one synthetic model, timed like the
    headline line (CUDA events on the model stream, inputs resident).  Returns the model's throughput keys."""
    import torch
    hm = synth.HostModel(cfg, seed)
    m = af.Model(cfg, [torch.from_numpy(b).to(dev) for b in hm.layers], torch.from_numpy(hm.token_embd).to(dev),
                 torch.from_numpy(hm.output_norm).to(dev), torch.from_numpy(hm.output).to(dev), max_chunk=C)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    stream = torch.cuda.ExternalStream(af.af_model_stream(m.h))
    prompt_dev = torch.from_numpy(hm.prompt(P)).to(dev)
    logits = torch.empty(cfg.n_vocab, dtype=torch.float32, device=dev)

    def one_step(ev):
        ev[0].record(stream)
        for p in range(0, P, C):
            n = min(C, P - p)
            af.af_prefill_dev(m.h, prompt_dev[p:p + n], n, p, logits if p + n >= P else None)
        ev[1].record(stream)
        for i in range(ND):
            af.af_decode_step(m.h, -1, P + i, logits)
        ev[2].record(stream)

    for _ in range(warmup):
        one_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for k in range(steps):
        one_step(evs[k])
    torch.cuda.synchronize()
    pre_s = sum(e[0].elapsed_time(e[1]) for e in evs) / 1000
    dec_s = sum(e[1].elapsed_time(e[2]) for e in evs) / 1000
    m.close()
    del m
    torch.cuda.empty_cache()
    dec_gbs = sum(decode_bytes_per_token(cfg, P + i) for i in range(ND)) * steps / dec_s / 1e9
    pf_tflops = prefill_flops(cfg, P, C)[0] * steps / pre_s / 1e12
    cpu_line = oracle_baselines(hm, cfg) if cpu else None
    del hm
    return {"cpu_baseline": cpu_line, "workload": f"{cfg.name}: {P}-token prompt in {C}-token chunks + {ND} greedy decode steps "
                        f"from position {P}, KV {cfg.kv_dtype} max_ctx {cfg.max_ctx}",
            "weights": cfg.wtype + (f" + {cfg.head_wtype} head" if cfg.head_wtype != cfg.wtype else ""),
            "seed": seed, "steps": steps, "warmup": warmup,
            "decode_tok_s": ND * steps / dec_s, "prefill_tok_s": P * steps / pre_s,
            "decode_hbm_gbs": dec_gbs, "decode_hbm_frac": dec_gbs / hbm_peak,
            "prefill_tflops": pf_tflops, "prefill_tc_frac": pf_tflops / tc_peak}


def kquant_run(af, args, dev, hbm_peak, tc_peak, steps=2, warmup=1):
    """Prefill + greedy decode of the 8B shape with Q4_K layers and a Q6_K head, timed like the main line."""
    cfg = synth.KQUANT_CONFIGS[1]
    out = workload_run(af, cfg, synth.kquant_seed_of(1), args.prompt, args.decode, args.chunk, dev, hbm_peak,
                       tc_peak, steps, warmup)
    gu = qgemv_roofline(af, cfg, dev, hbm_peak)
    head = qgemv_roofline(af, cfg, dev, hbm_peak, wtype=cfg.head_wtype, shape=(cfg.n_vocab, cfg.n_embd),
                          label="LM head")
    out["gemv_rooflines"] = [gu, head]
    return out


def workload_prompt(cfg):
    """Prompt tokens of a config's workload.  Where the prompt and the decode steps do not both fit the stated cache
    (the TinyLlama-shaped config: a 2048-token prompt and 128 decode steps at max_ctx 2048), the cache size is kept
    and the prompt is shortened so that the last decode step writes the last slot."""
    return min(cfg.prompt_len, cfg.max_ctx - cfg.n_decode)


def config_runs(af, args, dev, hbm_peak, tc_peak):
    """Every other full-size config over its own workload (the headline config is the main line)."""
    out = {}
    for idx in [int(x) for x in args.configs.split(",") if x.strip()]:
        if idx == args.config:
            continue
        cfg = synth.CONFIGS[idx]
        try:
            P = workload_prompt(cfg)
            line = workload_run(af, cfg, synth.seed_of(idx), P, cfg.n_decode, cfg.chunk, dev, hbm_peak,
                                tc_peak, steps=1, warmup=1, cpu=args.rank == 0 and not args.no_cpu_baseline)
            if cfg.max_ctx > 8192:  # long context: decode attention is half the bytes of a token; its roofline
                line["attn_roofline"] = attn_roofline(af, cfg, cfg.prompt_len, dev, hbm_peak)
            out[cfg.name] = line
            if cfg.max_ctx > 8192:  # the same workload over a Q8_0 cache with a 512-slot fp16 window
                qcfg = cfg.with_(kv_dtype="q8_0", kv_window=512)
                out[cfg.name + "+kv_q8_0"] = workload_run(af, qcfg, synth.seed_of(idx), P, cfg.n_decode, cfg.chunk,
                                                           dev, hbm_peak, tc_peak, steps=1, warmup=1)
        except Exception as e:  # a failed secondary line must not take the headline with it
            out[cfg.name] = {"error": f"{type(e).__name__}: {e}"}
    return out


def attn_roofline(af, cfg, pos, dev, hbm_peak, copies=4, reps=10):
    """Decode attention of one layer at position pos (the config's KV shape and dtype): algorithmic bytes
    2 * KVH * D * (pos + 1) * elem per launch over CUDA-event time, from a CUDA graph of `copies` back-to-back launches
    of af_attention_decode_static over `copies` separate caches (each larger than L2)."""
    import torch
    H, KVH, D, ctx = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.max_ctx
    dt = torch.float16 if cfg.kv_dtype == "f16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    caches = [(torch.randn(KVH, ctx, D, device=dev, generator=g).to(dt),
               torch.randn(KVH, ctx, D, device=dev, generator=g).to(dt)) for _ in range(copies)]
    q = torch.randn(H * D, device=dev, generator=g)
    out = torch.empty(H * D, device=dev)
    kvt = af.KVTYPE[cfg.kv_dtype]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for k, v in caches:  # first call per device: address lookup, outside capture
            af.af_attention_decode_static(q, k, v, kvt, H, KVH, D, ctx, pos, out, s)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(gr, stream=s):
        for k, v in caches:
            af.af_attention_decode_static(q, k, v, kvt, H, KVH, D, ctx, pos, out, s)
    gr.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
        for _ in range(reps):
            gr.replay()
        b.record(s)
    b.synchronize()
    ms = a.elapsed_time(b) / (reps * copies)
    nbytes = 2 * KVH * D * (pos + 1) * (2 if cfg.kv_dtype == "f16" else 4)
    gbs = nbytes / (ms / 1000) / 1e9
    del caches
    torch.cuda.empty_cache()
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "traffic": None, "kernel": f"decode attention {H}/{KVH}x{D} {cfg.kv_dtype} at position {pos}: graph of "
                                       f"{copies} back-to-back launches over {copies} caches",
            "bytes_per_launch": nbytes, "us_per_launch": ms * 1000}


def qgemv_roofline(af, cfg, dev, hbm_peak, reps=20, copies=8, wtype=None, shape=None, label="gate|up"):
    """af_qgemv on the model's gate|up shape [2F, E] (or `shape` in `wtype`): algorithmic bytes / CUDA-event time
    per launch.

    As in the decode step: a CUDA graph of `copies` back-to-back launches (programmatic dependent launch), each
    over its own copy of the weights (copies x 66 MB, far larger than L2, so no launch finds its weights in L2),
    replayed `reps` times on the launching stream.  A single launch after an L2 flush is reported beside it
    (cold: it also pays the launch and ramp that back-to-back launches overlap)."""
    import torch
    wt = wtype or cfg.wtype
    N, K = shape or (2 * cfg.n_ff, cfg.n_embd)
    W = synth.matrix(wt, 7, synth.TID_TEST_BASE + 99, N, K)
    Wd = torch.from_numpy(W).to(dev)
    hs = [af.af_qweight_create(af.WTYPE[wt], Wd, N, K) for _ in range(copies)]
    del Wd
    x = torch.randn(K, device=dev)
    y = torch.empty(N, device=dev)
    s = torch.cuda.Stream()
    for h in hs:
        af.af_qgemv(h, x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        for h in hs:
            af.af_qgemv(h, x, y)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # replays run on the current stream
        a.record(s)
        for _ in range(reps):
            g.replay()
        b.record(s)
    b.synchronize()
    ms = a.elapsed_time(b) / (reps * copies)
    # cold: one launch after writing a buffer larger than L2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream()
    cold = []
    for i in range(reps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        af.af_qgemv(hs[0], x, y)
        e1.record(cur)
        e1.synchronize()
        if i >= 3:
            cold.append(e0.elapsed_time(e1))
    for h in hs:
        af.af_qweight_destroy(h)
    bpe = synth.BLOCK_BYTES[wt] / synth.BLOCK_ELEMS[wt]
    nbytes = N * K * bpe + K * 4 + N * 4
    gbs = nbytes / (ms / 1000) / 1e9
    cold_ms = float(np.mean(cold))
    traffic = gemv_traffic(wt, N, K)
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "traffic": traffic,
            "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, captured on the "
                               "same kernel sources (hash " + GEMV_TRAFFIC["sources_sha256_16"] + ")")
            if traffic else "not captured for these sources",
            "kernel": f"qgemv {wt} [{N}x{K}] {label}: graph of {copies} back-to-back launches over "
                      f"{copies} weight copies ({copies * N * K * bpe / 1e6:.0f} MB > L2)",
            "bytes_per_launch": nbytes, "us_per_launch": ms * 1000,
            "cold_us_per_launch": cold_ms * 1000, "cold_frac": nbytes / (cold_ms / 1000) / 1e9 / hbm_peak}


def sampler_time(af, cfg, dev, reps=20):
    """Device time of one af_sample over a vocabulary-sized logits vector (penalty 1.1 on 64 recent ids,
    temperature 0.8, top-p 0.95), from a CUDA graph of `reps` calls with distinct draws u: a host loop of
    single calls would time the host, not the kernel."""
    import torch
    logits = torch.randn(cfg.n_vocab, device=dev) * 3
    recent = torch.randint(0, cfg.n_vocab, (64,), dtype=torch.int32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        af.af_sample(logits, cfg.n_vocab, recent, 64, 1.1, 0.8, 0.95, 0.37, tok)
    torch.cuda.synchronize()
    g, s = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        for i in range(reps):
            af.af_sample(logits, cfg.n_vocab, recent, 64, 1.1, 0.8, 0.95, (i + 0.5) / reps, tok)
    g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(5):
        g.replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) * 1000 / (5 * reps)


def gemv_traffic(wtype, N, K):
    """ncu DRAM bytes per launch for this shape, or None once the kernel's sources differ from the captured ones."""
    import hashlib
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(ROOT, "gguf_quantized_transformer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    t = GEMV_TRAFFIC
    if h.hexdigest()[:16] != t["sources_sha256_16"] or (wtype, N, K) != (t["wtype"], t["N"], t["K"]):
        return None
    return t["bytes"]


def e2e_run(af, m, prompt, cfg, args):
    """Host-API run: prompt ids from pinned host memory, greedy ids back to the host every step."""
    import torch
    P, ND, C = args.prompt, args.decode, args.chunk
    host_prompt = torch.from_numpy(prompt).pin_memory()
    hp = host_prompt.numpy()
    logits = torch.empty(cfg.n_vocab, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for p in range(0, P, C):
        n = min(C, P - p)
        af.af_prefill(m.h, hp[p:p + n], n, p, logits if p + n >= P else None)
    tok = af.af_model_sync(m.h, want_next=True)  # first greedy token on the host
    t1 = time.perf_counter()
    for i in range(ND):
        tok = af.af_decode_step(m.h, tok, P + i, None, want_next=True)
    t2 = time.perf_counter()
    return {"value": ND / (t2 - t1), "unit": "tok/s", "prefill_tok_s": P / (t1 - t0),
            "h2d_bytes_per_step": P * 4 + ND * 4, "d2h_bytes_per_step": (ND + 1) * 4,
            "note": "af_prefill from pinned host ids until the first greedy id is on the host, then "
                    "af_decode_step with the host feeding back each greedy id it reads (one stream sync per "
                    "token); wall clock"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--prompt", type=int, default=0, help="prompt tokens (default: the config's)")
    ap.add_argument("--decode", type=int, default=0, help="decode steps (default: the config's)")
    ap.add_argument("--chunk", type=int, default=512)
    ap.add_argument("--ref-decode", type=int, default=2, help="oracle decode steps per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kquant", action="store_true", help="skip the secondary Q4_K_M line")
    ap.add_argument("--configs", default="1,2,4", help="other configs to run over their own workloads ('' = none)")
    args = ap.parse_args()
    cfg = synth.CONFIGS[args.config]
    args.prompt = args.prompt or cfg.prompt_len
    args.decode = args.decode or cfg.n_decode
    world, rank, local = dist_setup()
    args.rank = rank
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
    else:
        run_ours(args, cfg, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
