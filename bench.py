"""Benchmark of the GB300 block-diffusion decoder (one JSON line on rank 0).

Workload: the full synthetic decoder (30 layers, d_model 2816, 16/8 heads of
128, 128 experts top-8 with FFN 704, vocab 262144, seeded random-init bf16
weights), a 2048-token uniform-random prompt, 4 canvases of 256 tokens,
denoising budget N = 48, adaptive stopping on, no EOS.

One step = the decode of all 4 canvases from the cached prompt, each canvas
denoised by the device-side loop (dg_denoise_canvas): every denoising forward (embed, 30 x {RMSNorm, QKV+RoPE, canvas attention, o-proj,
RMSNorm, router, routing (top-k + sort by expert), row gather, fused expert
FFN, combine}, final norm,
LM head fused with the vocab reduction, sampler) plus the 3 KV-append
forwards between canvases.  The prompt is encoded once before timing
(decode-only, as the pages measure); each step rewinds to it and uses a new
sample seed.  value = denoise steps/s (Eq. 8 total steps / time); output
tokens/s and TPF (Eq. 7, 10) are reported beside it.

The same JSON line also carries, each timed on the device with CUDA events:
the prompt encoding (prefill) of that workload; the kernel micro-ops at the
attention shapes (256 canvas queries, 16/4 heads of 128, prefix 0 / 1k / 8k /
32k keys), the MoE layer and LM head + sampler shapes (256 tokens, 128
experts top-8, vocab 262144) and the all-layer KV append; and the long
context workload (32768-token prompt, 16 canvases of 256, N = 48, paged KV);
and 4 such requests decoded in lockstep batches.
"""
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

METRIC = "denoise steps/s and output tokens/s per 256-token canvas on 1 GB300; % roofline"
PROMPT, CANVASES, BUDGET, C = 2048, 4, 48, 256
WORKLOAD = ("full synthetic decoder (30 layers, d_model 2816, 16/8 heads x 128, 128 experts top-8, "
            "FFN 704, vocab 262144), 2048-token random prompt, 4 canvases of 256, N=48, adaptive")


T_START = time.perf_counter()
VERBOSE = os.environ.get("DG_BENCH_VERBOSE") == "1"


def log(msg):
    """Progress of the run on stderr (the JSON line alone goes to stdout)."""
    print(f"[bench {time.perf_counter() - T_START:7.1f}s] {msg}", file=sys.stderr, flush=True)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(os.environ.get("DG_BENCH_BACKEND", "nccl"))
        pg = dist
    return world, rank, local, pg


def reduce_over_ranks(pg, value, op, device=None):
    """Barrier, then max or sum of `value` over ranks (identity on one rank)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.barrier()
    pg.all_reduce(t, op=pg.ReduceOp.MAX if op == "max" else pg.ReduceOp.SUM)
    return float(t.item())


# ---- CPU oracle sample (the reference arm and the cpu_baseline leg) ----------

class OracleSample:
    """A bounded slice of one denoising step of the workload, run by the oracle.

    One decoder layer over the 256-token canvas with a 2048-token prefix
    (attention + MoE over all experts the routing touches) and the LM head +
    sampler for 8 canvas positions.  Estimated step time = 30 x layer +
    32 x head(8 positions).  Weights are generated before timing.
    """

    def __init__(self, head_rows=8):
        import numpy as np
        from oracle import model as om, weights as ow
        self.np, self.om = np, om
        cfg = self.cfg = om.FULL
        s, std = cfg.weight_seed, cfg.init_std
        d, E, F = cfg.d_model, cfg.n_experts, cfg.d_ff
        qd, kd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
        t = lambda w: ow.layer_tid(0, w)
        self.W = dict(wq=ow.tensor(s, t(ow.WQ), (qd, d), std), wk=ow.tensor(s, t(ow.WK), (kd, d), std),
                      wv=ow.tensor(s, t(ow.WV), (kd, d), std), wo=ow.tensor(s, t(ow.WO), (d, qd), std),
                      wr=ow.tensor(s, t(ow.WR), (E, d), std), wg=ow.tensor(s, t(ow.WG), (E, F, d), std),
                      wu=ow.tensor(s, t(ow.WU), (E, F, d), std), wd=ow.tensor(s, t(ow.WD), (E, d, F), std),
                      attn_norm=np.ones(d), moe_norm=np.ones(d))
        self.lm_head = ow.tensor(s, ow.LM_HEAD, (cfg.vocab, d), std)
        rng = np.random.default_rng(0)
        ids = rng.integers(0, cfg.vocab, C)
        self.h = ow.rows(s, ow.EMBED, (cfg.vocab, d), ids, std).astype(np.float64)
        self.pk = rng.standard_normal((PROMPT, cfg.n_kv_heads, cfg.head_dim)) * 0.5
        self.pv = rng.standard_normal((PROMPT, cfg.n_kv_heads, cfg.head_dim)) * 0.5
        self.head_rows = head_rows
        self.threads = os.cpu_count()

    def run(self):
        """Returns the estimated seconds of one full denoising step."""
        np, om, cfg = self.np, self.om, self.cfg
        from oracle import sampler as osamp
        pos = PROMPT + np.arange(C)
        t0 = time.perf_counter()
        h, _, _ = om.block(self.h, pos, self.W, cfg, self.pk, self.pv, "bidir")
        t1 = time.perf_counter()
        n = om.rmsnorm(h[: self.head_rows], 1.0, cfg.rms_eps)
        l = np.empty((self.head_rows, cfg.vocab), np.float32)
        for v0 in range(0, cfg.vocab, 32768):
            l[:, v0:v0 + 32768] = n @ self.lm_head[v0:v0 + 32768].astype(np.float64).T
        osamp.position_outputs(l, 1, 0, 1)
        t2 = time.perf_counter()
        return cfg.n_layers * (t1 - t0) + (C / self.head_rows) * (t2 - t1)

    def describe(self):
        return (f"oracle (numpy fp64 forward + fp32 sampler) on layer 0 of a denoising step "
                f"(256-token canvas, {PROMPT}-token prefix, MoE over the experts its routing picks, "
                f"~120 of 128 in layer 0 vs ~15 in deep layers, so 30 x layer overstates the oracle's "
                f"step time) and the LM head + sampler for {self.head_rows} positions; "
                f"step time = 30 x layer + {C // self.head_rows} x head")


def reference_arm(args):
    world, rank, local, pg = dist_setup()
    if rank != 0:
        return 0
    smp = OracleSample()
    for _ in range(args.warmup):
        smp.run()
    walls, est = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        est.append(smp.run())
        walls.append(time.perf_counter() - t0)
    step_s = sum(est) / len(est)
    v = 1.0 / step_s
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "denoise steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sum(walls) / len(walls) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "step": ("a bounded sample of one denoising step (one layer + 8 LM-head rows); "
                                "ms_per_step is the sample's measured wall time, value the denoising "
                                "steps/s of the full step it extrapolates to")},
            "estimated_ms_per_full_step": step_s * 1e3,
            "cpu_baseline": {"value": v, "unit": "denoise steps/s", "cores": smp.threads,
                             "kind": "oracle", "sample": smp.describe()},
            "e2e": {"value": v, "unit": "denoise steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- the GPU arm -------------------------------------------------------------

def decode_all(dgp, m, seed, scfg):
    """One bench step: rewind to the prompt and decode all canvases."""
    dgp.dg_rewind(m, PROMPT)
    scfg.sample_seed = seed
    dgp.dg_set_sampler(m, scfg)
    Ns, Cs = [], []
    for k in range(CANVASES):
        Ns.append(dgp.dg_denoise_canvas(m))          # device-side loop: one sync per canvas
        if VERBOSE:
            log(f"canvas {k}: {Ns[-1]} steps")
        if k < CANVASES - 1:
            _, valid = dgp.dg_commit_canvas(m)
        else:
            valid = C
        Cs.append(valid)
    return Ns, Cs


# DRAM traffic / algorithmic bytes of the decoder's own expert-FFN launches:
# dram__bytes_read.sum + dram__bytes_write.sum of all 30 launches of one eager
# denoising step (ncu, 1 pass, `python bench.py --profile-step` with routing
# and scatter unfused), over their algorithmic bytes from the same step's
# experts touched (profiles/launch_list_full_decoder.md).  Below 1: the
# weights stream once and part of the row, SwiGLU and output bytes stay in L2.
FFN_TRAFFIC_RATIO = 7.951e9 / 8.717e9


def expert_bytes(cfg, experts_per_launch, rows_per_launch):
    """Algorithmic DRAM bytes of one expert-FFN launch (gate/up, SwiGLU and
    down of every routed expert): the gate/up and down weights of every expert
    that received a row, once (the count is measured on the device by the
    routing kernel), the gathered token rows, the SwiGLU activations written
    and read back, and the bf16 outputs."""
    d, F = cfg.d_model, cfg.d_ff
    e, r = experts_per_launch, rows_per_launch
    return {"expert_ffn": e * 3 * F * d * 2 + r * d * 2 + 2 * r * F * 2 + r * d * 2}


def gpu_arm(args):
    import numpy as np
    import torch
    import discrete_diffusion_block_gb300 as dgp
    from discrete_diffusion_block_gb300 import build, synth

    world, rank, local, pg = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if pg is not None:
        pg.barrier()
    dgp.load()
    hbm, tf_burst, tf_sust, peak_src = peaks()

    stream = torch.cuda.Stream(device=dev)
    cfg = dgp.full_config(max_context=PROMPT + CANVASES * C, n_layers=args.layers)
    scfg = dgp.SamplerConfig(budget_N=BUDGET, adaptive=1)
    m = dgp.dg_init_model(cfg, scfg, stream=stream)
    log("model initialised")
    prompt = synth.prompt_ids(PROMPT, cfg.vocab, seed=1000 + rank)
    dgp.dg_prefill(m, prompt)                       # first call: kernel attributes, tensor maps
    prefill = time_prefill(dgp, m, prompt, stream, cfg, tf_burst)
    log("prefill timed")

    for w in range(args.warmup):
        decode_all(dgp, m, 10_000 + w, scfg)
        log(f"warm-up decode {w + 1} of {args.warmup}")

    # ---- timed region: the value (launch counting only, no per-kernel events)
    dgp.dg_profile(m, 2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    allN, allC = [], []
    rdev = dev if pg is not None else None
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        ev0.record(stream)
        for s in range(args.steps):
            Ns, Cs = decode_all(dgp, m, 20_000 + s, scfg)
            allN += Ns
            allC += Cs
        ev1.record(stream)
        torch.cuda.synchronize()
    launches = int(sum(n for _, n in dgp.dg_profile_read(m).values()))
    ms = ev0.elapsed_time(ev1)
    log(f"timed region: {args.steps} decodes in {ms:.0f} ms")
    ms_max = reduce_over_ranks(pg, ms, "max", rdev)
    steps_total = reduce_over_ranks(pg, sum(allN), "sum", rdev)
    tokens_total = reduce_over_ranks(pg, sum(allC), "sum", rdev)
    value = steps_total / (ms_max / 1e3)
    tok_s = tokens_total / (ms_max / 1e3)
    tpf = sum(allC) / (sum(allN) + args.steps * (CANVASES - 1))
    eff = sum(n * c for n, c in zip(allN, allC)) / max(sum(allC), 1)

    # ---- profiled step: CUDA events around every kernel (graph event nodes) ----
    dgp.dg_profile(m, 1)
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record(stream)
    pN, _ = decode_all(dgp, m, 40_000, scfg)
    pe1.record(stream)
    torch.cuda.synchronize()
    prof = dgp.dg_profile_read(m)
    touched, routed = dgp.dg_profile_experts(m)
    dgp.dg_profile(m, 0)
    log("profiled decode done")
    n_moe = max(prof["expert_ffn"][1], 1)                    # one expert-FFN launch per MoE layer
    per_launch = expert_bytes(cfg, touched / n_moe, routed / n_moe)
    hbm, tf_burst, tf_sust, peak_src = peaks()
    kernels = {}
    for name, (kms, n) in prof.items():
        if n:
            kernels[name] = {"ms_total": round(kms, 3), "launches": n,
                             "us_per_launch": round(kms / n * 1e3, 2)}
    for name, b in per_launch.items():
        if prof[name][1] and prof[name][0] > 0:
            a = b / (prof[name][0] / 1e3 / prof[name][1]) / 1e9
            kernels[name].update(GBps=round(a, 1), frac_hbm=round(a / hbm, 4))
    if prof["lm_head"][1] and prof["lm_head"][0] > 0:
        # the method's work, 2 C d V flops; the kernel issues two MMAs per weight
        # tile (hi and lo bf16 halves of the fp32 final-norm rows), twice that
        fl = 2.0 * C * cfg.d_model * cfg.vocab
        a = fl / (prof["lm_head"][0] / 1e3 / prof["lm_head"][1]) / 1e12
        kernels["lm_head"].update(TFLOPs=round(a, 1), frac_bf16_sustained=round(a / tf_sust, 4),
                                  flops_per_launch=fl, mma_flops_per_launch=2 * fl,
                                  note="TFLOPs on the method's 2*C*d*V; the hi/lo split issues 2x that in MMAs")
    # the dominant kernel class of the step with a roofline: the expert FFN
    # (HBM-bound weight streaming) or the LM head (tensor-bound contraction)
    measured_in = (f"profiled step after the timed region ({pe0.elapsed_time(pe1):.0f} ms, "
                   f"{sum(pN)} denoising steps)")
    if prof["lm_head"][0] > prof["expert_ffn"][0] and "TFLOPs" in kernels.get("lm_head", {}):
        kms, n = prof["lm_head"]
        fl = 2.0 * C * cfg.d_model * cfg.vocab
        achieved = fl / (kms / 1e3 / n) / 1e12
        roofline = {"kernel": "lm_head", "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": tf_sust, "unit": "TFLOP/s", "frac": round(achieved / tf_sust, 4),
                    "traffic": args.traffic, "peak_source": f"{peak_src} bf16_tflops_sustained",
                    "algorithmic_flops_per_launch": fl, "measured_in": measured_in}
    else:
        dom = "expert_ffn"
        kms, n = prof[dom]
        achieved = per_launch[dom] / (kms / 1e3 / n) / 1e9
        traffic = args.traffic if args.traffic is not None else round(FFN_TRAFFIC_RATIO * per_launch[dom])
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                    "traffic_source": ("ncu dram bytes / algorithmic bytes of the 30 expert-FFN launches of one "
                                       f"eager decoder step ({FFN_TRAFFIC_RATIO:.3f}), times this launch's algorithmic bytes"),
                    "peak_source": f"{peak_src} hbm_gbs",
                    "algorithmic_bytes_per_launch": round(per_launch[dom]), "measured_in": measured_in}

    # ---- e2e through the public API: host prompt in, host ids out ----------
    e2e = None
    if args.e2e_steps > 0:
        dgp.dg_set_sampler(m, dgp.SamplerConfig(budget_N=BUDGET, adaptive=1, sample_seed=30_000))
        host_prompt = np.ascontiguousarray(prompt, dtype=np.int32)
        t0 = time.perf_counter()
        e_steps, h2d, d2h = 0, 0, 0
        for s in range(args.e2e_steps):
            out, st = dgp.dg_generate(m, host_prompt, CANVASES)
            e_steps += st["total_steps"]
            h2d += host_prompt.nbytes
            d2h += out.nbytes + 4 * st["total_steps"]     # canvases + one done flag per step
        el = time.perf_counter() - t0
        e2e = {"value": e_steps / el, "unit": "denoise steps/s",
               "h2d_bytes_per_step": h2d // args.e2e_steps, "d2h_bytes_per_step": d2h // args.e2e_steps,
               "calls": args.e2e_steps,
               "includes": "prefill of the 2048-token prompt + decode of 4 canvases per dg_generate call"}
    log("end-to-end calls done")
    m.close()
    del m

    micro_lines, long_ctx, batch, fp8 = None, None, None, None
    if rank == 0 and not args.no_extra:
        micro_lines = micro_results(dgp, "all", args.micro_reps)
        log("micro-ops done")
        long_ctx = long_context(dgp, stream, tf_burst)
        log("long context done")
        batch = batched(dgp, stream)
        log("batched done")
        fp8 = fp8_experts(dgp, stream, value)
        log("fp8 experts done")
    expert_gb = touched / n_moe * 3 * cfg.d_ff * cfg.d_model * 2 * cfg.n_layers / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample()
        est = smp.run()
        log("CPU baseline sample done")
        cpu = {"value": 1.0 / est, "unit": "denoise steps/s", "cores": smp.threads, "kind": "oracle",
               "sample": smp.describe()}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "denoise steps/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic: seeded random-init weights, uniform random prompt ids",
                "config": {"workload": WORKLOAD if args.layers == 30 else
                           WORKLOAD.replace("30 layers", f"{args.layers} layers (profiling case, not the headline)"),
                           "step": "decode of 4 canvases (all denoising steps + 3 KV-append forwards), prompt cached",
                           "l2": (f"inputs larger than L2 (129 MB): {expert_gb:.1f} GB of expert weights "
                                  f"({touched / n_moe:.1f} experts touched per MoE launch, measured) and "
                                  f"the 1.48 GB LM head streamed per denoising step"),
                           "parallelism": f"replicas x{world}"},
                "output_tokens_per_s": tok_s, "tpf": tpf, "effective_steps": eff,
                "N_k_mean": sum(allN) / len(allN),
                "experts_touched_per_moe_launch": round(touched / n_moe, 2),
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "prefill": prefill, "micro": micro_lines, "long_context": long_ctx, "batched": batch,
                "fp8_experts": fp8,
                "clocks": clk.summary(), "gpu_launches": launches}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


# ---- prefill, kernel micro-ops and the long-context workload ---------------------

def causal_attention_flops(n, prefix, Hq, hd):
    """Algorithmic flops of one layer's attention for n new tokens after
    `prefix` cached ones, causal inside the new block: 4 Hq hd per visible pair."""
    return 4.0 * Hq * hd * (n * prefix + n * (n + 1) / 2)


def time_prefill(dgp, m, prompt, stream, cfg, tf_burst, chunk=2048):
    """Device time of dg_prefill (events on the model's stream; the call also
    syncs after each chunk), then a second prefill with per-kernel events for
    the causal attention's rate."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dgp.dg_profile(m, 2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    dgp.dg_prefill(m, prompt)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dgp.dg_profile(m, 1)
    dgp.dg_prefill(m, prompt)
    prof = dgp.dg_profile_read(m)
    dgp.dg_profile(m, 0)
    n = len(prompt)
    fl = 0.0
    for p0 in range(0, n, chunk):      # the prompt is encoded in chunks; the last layer needs K/V only
        fl += (cfg.n_layers - 1) * causal_attention_flops(min(chunk, n - p0), p0, cfg.n_q_heads, cfg.head_dim)
    ams, al = prof["attention"]
    out = {"tokens": n, "ms": round(e0.elapsed_time(e1), 3), "wall_ms": round(wall * 1e3, 3),
           "tokens_per_s": round(n / (e0.elapsed_time(e1) / 1e3), 1)}
    if ams > 0:
        a = fl / (ams / 1e3) / 1e12
        out["attention"] = {"launches": al, "ms": round(ams, 3), "TFLOPs": round(a, 1),
                            "frac_bf16": round(a / tf_burst, 4), "flops": fl,
                            "note": "causal; flops count visible (query, key) pairs only"}
    out["kernels_ms"] = {k: round(v[0], 3) for k, v in prof.items() if v[1]}
    return out


def micro_results(dgp, which, reps):
    """Per-kernel timings at the micro-op shapes (median of `reps` L2-flushed runs)."""
    import numpy as np
    import torch
    from discrete_diffusion_block_gb300 import synth
    hbm, tf_burst, tf_sust, src = peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MB > L2

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts) / 1e3

    out = []
    if which in ("attention", "all"):
        Hq, Hkv, hd, C_, pg = 16, 4, 128, 256, 128
        for P in (0, 1024, 8192, 32768):
            S = P + C_
            n_pages = (S + pg - 1) // pg
            kp = torch.randn(n_pages, Hkv, pg, hd, device=dev).to(torch.bfloat16)
            vp = torch.randn(n_pages, Hkv, pg, hd, device=dev).to(torch.bfloat16)
            q = torch.randn(C_, Hq, hd, device=dev).to(torch.bfloat16)
            table = torch.arange(n_pages, dtype=torch.int32, device=dev)
            o = torch.empty_like(q)
            ws = torch.empty(max(dgp.dg_op_attention_workspace_bytes(P, C_, Hq, Hkv, hd), 1),
                             dtype=torch.uint8, device=dev)
            sec = timed(lambda: dgp.dg_op_canvas_attention(q, kp, vp, table, P, C_, Hq, Hkv, hd, pg,
                                                           False, o, ws))
            fl = 4.0 * C_ * Hq * S * hd
            log(f"micro attention P={P}")
            out.append({"micro": "canvas_attention", "shape": f"P={P} C={C_} Hq={Hq} Hkv={Hkv} hd={hd}",
                        "ms": sec * 1e3, "TFLOPs": fl / sec / 1e12, "frac_bf16": fl / sec / 1e12 / tf_burst})
            del kp, vp
    if which in ("moe", "all"):
        T, d, E, k, F = 256, 2816, 128, 8, 704
        wr = torch.empty(E * d, dtype=torch.bfloat16, device=dev)
        wgu = torch.empty(E * 2 * F * d, dtype=torch.bfloat16, device=dev)
        wd = torch.empty(E * d * F, dtype=torch.bfloat16, device=dev)
        dgp.dg_op_fill_moe_weights(wr, wgu, wd, d, E, F, 0, 0)
        _, xt = synth.normal_bf16((T, d), seed=3)
        x = xt.to(dev)
        y = torch.empty(T, d, dtype=torch.float32, device=dev)
        ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        gates = torch.empty(T, k, dtype=torch.float32, device=dev)
        ws = torch.empty(dgp.dg_op_moe_workspace_bytes(T, d, E, k, F), dtype=torch.uint8, device=dev)
        sec = timed(lambda: dgp.dg_op_moe(x, wr, wgu, wd, T, d, E, k, F, y, ids, gates, ws))
        touched = len(np.unique(ids.cpu().numpy()))
        byt = touched * 3 * F * d * 2 + E * d * 2
        fl = 2.0 * T * k * 3 * F * d
        log("micro moe")
        out.append({"micro": "moe_layer", "shape": f"T={T} d={d} E={E} top{k} F={F}",
                    "experts_touched": touched, "ms": sec * 1e3, "GBps": byt / sec / 1e9,
                    "frac_hbm": byt / sec / 1e9 / hbm, "TFLOPs": fl / sec / 1e12,
                    "includes": "route + scatter + expert FFN + combine"})
        del wr, wgu, wd
    if which in ("lmhead", "all"):
        T, d, V = 256, 2816, 262144
        w = torch.empty(V * d, dtype=torch.bfloat16, device=dev)
        dgp.dg_op_fill_tiled_weights(w, V, d, 0, 2)
        tiles = lambda t: torch.from_numpy(dgp.to_operand_tiles(t.view(torch.int16).numpy())).view(
            torch.bfloat16).to(dev)
        # the decoder's form first: an fp32 activation as a bf16 hi + lo pair
        xf = torch.from_numpy(synth.normal((T, d), seed=2))
        hi = xf.to(torch.bfloat16)
        lo = (xf - hi.float()).to(torch.bfloat16)
        x, x_lo = tiles(hi), tiles(lo)
        part = torch.empty(dgp.partials_bytes(T, V) // 4, dtype=torch.int32, device=dev)
        fl = 2.0 * T * d * V
        for name, xl in (("hi + lo bf16 activation, the decoder's form: 2x the MMAs", x_lo),
                         ("single bf16 activation", None)):
            sec = timed(lambda: dgp.dg_op_lm_head_partials(x, w, T, d, V, 1, 0, 1, part, xn_lo=xl))
            log("micro lm head")
            out.append({"micro": "lm_head_partials", "shape": f"T={T} d={d} V={V} ({name})",
                        "ms": sec * 1e3, "TFLOPs": fl / sec / 1e12, "frac_bf16": fl / sec / 1e12 / tf_burst,
                        "GBps_weights": V * d * 2 / sec / 1e9})
        del w
    if which in ("sampler", "all"):
        C_, V = 256, 262144
        logits = torch.from_numpy(synth.logits(C_, V, seed=1)).to(dev)
        part = torch.empty(dgp.partials_bytes(C_, V) // 4, dtype=torch.int32, device=dev)
        sc = dgp.SamplerConfig()
        st = [torch.zeros(C_, dtype=torch.int32, device=dev) for _ in range(6)]
        com = torch.zeros(C_, dtype=torch.uint8, device=dev)
        conf = torch.zeros(C_, dtype=torch.float32, device=dev)
        done = torch.zeros(1, dtype=torch.int32, device=dev)

        def run():
            dgp.dg_op_logits_partials(logits, C_, V, 1, 0, 1, part)
            dgp.dg_op_sampler_update(part, C_, V, 1, sc, st[0], com, st[1], st[2], st[3], conf, st[4], done)
        sec = timed(run)
        byt = C_ * V * 4
        log("micro sampler")
        out.append({"micro": "sampler_materialized_logits", "shape": f"C={C_} V={V}", "ms": sec * 1e3,
                    "GBps": byt / sec / 1e9, "frac_hbm": byt / sec / 1e9 / hbm})
        del logits
    if which in ("kv_append", "all"):
        L, n, Hkv, hd, pg = 30, 256, 8, 128, 128
        n_pages = 32
        kn = torch.randn(L, n, Hkv, hd, device=dev).to(torch.bfloat16)
        vn = torch.randn(L, n, Hkv, hd, device=dev).to(torch.bfloat16)
        kp = torch.zeros(L, n_pages, Hkv, pg, hd, dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        table = torch.arange(n_pages, dtype=torch.int32, device=dev)
        sec = timed(lambda: dgp.dg_op_kv_append(kn, vn, kp, vp, table, L, n_pages, 2048, n, Hkv, hd, pg))
        byt = 2 * 2 * L * n * Hkv * hd * 2
        out.append({"micro": "kv_append", "shape": f"layers={L} tokens={n} Hkv={Hkv} hd={hd}",
                    "ms": sec * 1e3, "GBps": byt / sec / 1e9, "frac_hbm": byt / sec / 1e9 / hbm})
    for o in out:
        o["peak_source"] = src
        for k in ("ms", "TFLOPs", "GBps", "GBps_weights"):
            if k in o:
                o[k] = round(o[k], 4 if k == "ms" else 1)
        for k in ("frac_bf16", "frac_hbm"):
            if k in o:
                o[k] = round(o[k], 4)
    del flush
    torch.cuda.empty_cache()
    return out


LONG_PROMPT, LONG_CANVASES = 32768, 16


def long_context(dgp, stream, tf_burst):
    """The long-context workload: 32768-token random prompt, 16 canvases of
    256, N = 48, adaptive stopping, paged KV cache (pages of 128 tokens).
    One decode of all canvases, timed with CUDA events on the model's
    stream, after one untimed decode of the first canvas (graph capture)."""
    import torch
    from discrete_diffusion_block_gb300 import synth
    cfg = dgp.full_config(max_context=LONG_PROMPT + LONG_CANVASES * C)
    scfg = dgp.SamplerConfig(budget_N=BUDGET, adaptive=1, sample_seed=50_000)
    m = dgp.dg_init_model(cfg, scfg, stream=stream)
    prompt = synth.prompt_ids(LONG_PROMPT, cfg.vocab, seed=77)
    dgp.dg_prefill(m, prompt)
    log("long context: prefill done")
    prefill = time_prefill(dgp, m, prompt, stream, cfg, tf_burst)
    log("long context: prefill timed")
    Ns, Cs = [], []
    dgp.dg_profile(m, 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for k in range(LONG_CANVASES):
        Ns.append(dgp.dg_denoise_canvas(m))
        log(f"long context: canvas {k} ({Ns[-1]} steps)")
        if k < LONG_CANVASES - 1:
            _, valid = dgp.dg_commit_canvas(m)
        else:
            valid = C
        Cs.append(valid)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    launches = int(sum(n for _, n in dgp.dg_profile_read(m).values()))
    m.close()
    del m
    torch.cuda.empty_cache()
    steps, tok = sum(Ns), sum(Cs)
    return {"workload": (f"{LONG_PROMPT}-token random prompt, {LONG_CANVASES} canvases of {C}, N={BUDGET}, "
                         "adaptive, paged KV (128-token pages), same decoder"),
            "denoise_steps_per_s": round(steps / (ms / 1e3), 2),
            "output_tokens_per_s": round(tok / (ms / 1e3), 1),
            "decode_ms": round(ms, 1), "total_steps": steps, "total_tokens": tok,
            "effective_steps_eq9": round(sum(n * c for n, c in zip(Ns, Cs)) / tok, 3),
            "tpf_eq10": round(tok / (steps + LONG_CANVASES - 1), 3), "N_k": Ns,
            "prefill": prefill, "gpu_launches": launches,
            "note": "decode from the cached prompt, first canvas included (its CUDA graphs are captured on the fly)"}


BATCH = 4


def fp8_experts(dgp, stream, bf16_value):
    """The same workload as the value (2048-token prompt, 4 canvases of 256,
    N = 48, adaptive) with the experts' gate/up products in FP8 e4m3
    (dg_config.expert_fp8): two untimed decodes (graph capture, warm-up), then
    two decodes timed with CUDA events on the model's stream.  Not the
    headline: the value is the bf16 decoder's."""
    import torch
    from discrete_diffusion_block_gb300 import synth
    cfg = dgp.full_config(max_context=PROMPT + CANVASES * C, expert_fp8=1)
    scfg = dgp.SamplerConfig(budget_N=BUDGET, adaptive=1)
    m = dgp.dg_init_model(cfg, scfg, stream=stream)
    dgp.dg_prefill(m, synth.prompt_ids(PROMPT, cfg.vocab, seed=1000))
    for w in range(2):
        decode_all(dgp, m, 20_000 + w, scfg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    Ns = []
    for s in range(2):
        n, _ = decode_all(dgp, m, 30_000 + s, scfg)
        Ns += n
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    m.close()
    del m
    torch.cuda.empty_cache()
    value = sum(Ns) / (ms / 1e3)                 # counted like the value: denoising steps (Eq. 8)
    return {"workload": WORKLOAD + "; expert gate/up products in FP8 e4m3 (per-row power-of-two scales)",
            "denoise_steps_per_s": round(value, 2), "vs_bf16_experts": round(value / bf16_value, 3),
            "decode_ms": round(ms, 1), "N_k": Ns,
            "note": "W_down and the SwiGLU output stay bf16; timed like the value (all canvases of a "
                    "decode, KV-append forwards included; denoising steps counted)"}


def batched(dgp, stream):
    """Lockstep multi-request batching on the same decoder: 4 requests, each a
    2048-token random prompt and 4 canvases of 256 (N = 48, adaptive), every
    forward over all 4 canvases.  One decode of all canvases from the cached
    prompts, timed with CUDA events on the model's stream (after one untimed
    decode that captures the graphs)."""
    import torch
    from discrete_diffusion_block_gb300 import synth
    cfg = dgp.full_config(max_context=PROMPT + CANVASES * C, max_requests=BATCH)
    scfg = dgp.SamplerConfig(budget_N=BUDGET, adaptive=1, sample_seed=60_000)
    m = dgp.dg_init_model(cfg, scfg, stream=stream)
    prompts = [synth.prompt_ids(PROMPT, cfg.vocab, seed=3000 + b) for b in range(BATCH)]

    def decode():
        dgp.dg_prefill_batch(m, prompts)
        Ns = []
        for k in range(CANVASES):
            Ns.append(dgp.dg_denoise_canvas_batch(m))
            if k < CANVASES - 1:
                dgp.dg_commit_canvas_batch(m)
        return Ns
    decode()
    dgp.dg_prefill_batch(m, prompts)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    Ns = []
    for k in range(CANVASES):
        Ns.append(dgp.dg_denoise_canvas_batch(m))
        if k < CANVASES - 1:
            dgp.dg_commit_canvas_batch(m)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    m.close()
    del m
    torch.cuda.empty_cache()
    steps = sum(sum(n) for n in Ns)                 # per-request steps (Eq. 8 summed over requests)
    forwards = sum(max(n) for n in Ns)              # lockstep forwards over all 4 canvases
    tokens = BATCH * CANVASES * C
    return {"workload": (f"{BATCH} requests in lockstep on the same decoder, each a {PROMPT}-token random "
                         f"prompt and {CANVASES} canvases of {C}, N={BUDGET}, adaptive"),
            "requests": BATCH, "decode_ms": round(ms, 1),
            "denoise_steps_per_s": round(steps / (ms / 1e3), 2),
            "output_tokens_per_s": round(tokens / (ms / 1e3), 1),
            "batched_forwards": forwards, "ms_per_batched_step": round(ms / (forwards + CANVASES - 1), 3),
            "N_k_per_request": [[n[b] for n in Ns] for b in range(BATCH)],
            "note": "requests' steps summed; a batched forward serves every request's canvas"}


def profile_step(args):
    """--profile-step: the decoder of the value, its prompt encoded, then one
    eager denoising step (every kernel of a step launched directly, none from
    a graph) -- the command profilers capture; prints one short line."""
    import torch
    import discrete_diffusion_block_gb300 as dgp
    from discrete_diffusion_block_gb300 import build, synth
    torch.cuda.set_device(0)
    build.build()
    dgp.load()
    stream = torch.cuda.Stream(device=torch.device("cuda", 0))
    cfg = dgp.full_config(max_context=PROMPT + CANVASES * C, n_layers=args.layers)
    m = dgp.dg_init_model(cfg, dgp.SamplerConfig(budget_N=BUDGET, adaptive=1), stream=stream)
    dgp.dg_prefill(m, synth.prompt_ids(PROMPT, cfg.vocab, seed=1000))
    torch.cuda.synchronize()
    dgp.dg_denoise_step(m)
    torch.cuda.synchronize()
    import numpy as np
    touched = [int(len(np.unique(dgp.dg_read_routing(m, L)))) for L in range(cfg.n_layers)]
    per_expert = 3 * cfg.d_ff * cfg.d_model * 2
    rows = C * cfg.top_k
    fixed = rows * cfg.d_model * (2 + 4) + rows * cfg.d_ff * 2 * 2     # rows in, y out, SwiGLU out + in
    print(json.dumps({"profile_step": "done", "layers": cfg.n_layers, "experts_touched": touched,
                      "expert_ffn_algorithmic_bytes": [e * per_expert + fixed for e in touched]}), flush=True)
    m.close()
    return 0


def micro(args):
    """--micro: the kernel micro-ops only, one JSON line per case."""
    import torch
    import discrete_diffusion_block_gb300 as dgp
    from discrete_diffusion_block_gb300 import build
    torch.cuda.set_device(0)
    build.build()
    dgp.load()
    for o in micro_results(dgp, args.micro, args.steps):
        print(json.dumps(o), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the micro-op and long-context sections of the JSON line")
    ap.add_argument("--micro-reps", type=int, default=10)
    ap.add_argument("--section", default=None, choices=["long", "batched", "fp8"],
                    help="run one extra section of the JSON line alone and print it")
    ap.add_argument("--micro", default=None,
                    choices=["moe", "lmhead", "sampler", "attention", "kv_append", "all"],
                    help="kernel micro-benchmarks at the micro-op shapes instead of the decoder")
    ap.add_argument("--layers", type=int, default=30,
                    help="decoder depth; fewer layers give a small case of the same kernels for ncu captures")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, if measured for the current binaries")
    ap.add_argument("--profile-step", action="store_true",
                    help="prefill + one eager denoising step of the decoder (for profiler captures)")
    args = ap.parse_args()
    if args.profile_step:
        return profile_step(args)
    if args.micro:
        return micro(args)
    if args.section:
        import torch
        import discrete_diffusion_block_gb300 as dgp
        from discrete_diffusion_block_gb300 import build
        torch.cuda.set_device(0)
        build.build()
        dgp.load()
        stream = torch.cuda.Stream(device=torch.device("cuda", 0))
        if args.section == "long":
            out = long_context(dgp, stream, peaks()[1])
        elif args.section == "batched":
            out = batched(dgp, stream)
        else:
            out = fp8_experts(dgp, stream, float("nan"))
        print(json.dumps(out), flush=True)
        return 0
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
