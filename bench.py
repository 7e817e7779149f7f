#!/usr/bin/env python3
"""Benchmark of the Q4_K weight-only hot path on GB300.

Headline (one JSON line on rank 0): the 27B-shape hybrid decode step, batch 1
(64 layers: 48 Gated-DeltaNet + 16 full-attention projection sets, d_model
5120, SwiGLU 17408, Q8_0 lm_head over 248320 tokens, argmax; ~15.05 GB of
weights per token) as ONE kernel launch per token, in tokens/s.  The same line
carries the roofline of that launch against measured HBM bandwidth, the
end-to-end number through the C ABI with the token crossing host<->device
every step, the CPU oracle timed on this host, the SM clocks seen during the
timed region, and component results: the single 5120x5120 Q4_K GEMV, the
batch-1 MLP and its batched-GEMV sweep, the prefill GEMMs and the GEMV shape
sweep with one-launch vs per-matmul decode.

Weights are synthetic (seeded N(0, 0.02^2) f32 quantized to Q4_K / Q8_0 on
the GPU; embedding N(0, 1)); they are larger than L2, so no flush is needed
for the decode.  Multi-GPU runs (torchrun) are independent replicas: the
decode step does not shard, each rank decodes its own stream.

  python bench.py [--steps K] [--warmup W] [--quick] [--impl reference]

Profiling cases (not the headline): --layers L and --vocab V shrink the decode
stack (the weights per token and the model shape change accordingly, and the
line's config says so); --components picks the component sections to run.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_K GEMV GB/s (% HBM peak); 27B-shape decode-step tok/s; prefill TFLOPS"
D, F, V, GI, QG, KV, NM, NL = 5120, 17408, 248320, 16480, 12288, 1024, 6144, 64
SEED_DECODE = 3
COMPONENTS = ("gemv", "mlp", "batch", "prefill", "mixer", "prefill_forward")
# the mixer bodies of the 27B shape: GDN 16 key / 48 value heads of 128, FA 24 query / 4 KV heads of 256
MIX = dict(gdn_nk=16, gdn_nv=48, fa_nq=24, fa_nkv=4, fa_rot=64, rope_theta=1e7, eps=1e-6)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only, no component sections")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--layers", type=int, default=NL, help="decode stack depth (profiling cases only)")
    ap.add_argument("--vocab", type=int, default=V, help="lm_head rows (profiling cases only)")
    ap.add_argument("--components", default="all",
                    help="comma list of gemv,mlp,batch,prefill, or 'all' / 'none'")
    a = ap.parse_args()
    if a.quick:
        a.components = "none"
    a.components = set(COMPONENTS) if a.components == "all" else (
        set() if a.components == "none" else set(a.components.split(",")))
    bad = a.components - set(COMPONENTS)
    if bad:
        ap.error("unknown components: %s" % ",".join(sorted(bad)))
    if a.vocab < 1 or a.layers < 1:
        ap.error("--layers and --vocab must be positive")
    return a


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)) or None, \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs.  The sampler is
    started first and the region begins only once its first sample has arrived (nvidia-smi takes a moment
    to start), every 25 ms; the summary counts the samples that arrived inside the region, and at least the
    first one after its start when the region is shorter than the interval."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.first = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.last = len(self.lines)
        if self.proc:
            time.sleep(0.06)  # the sample that straddles the region's end
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = self.lines[self.first:max(self.last, self.first + 1)]
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------------ model on the device
def q4k_device(fak, torch, seed, tid, n, k, scratch):
    """Generate W ~ N(0, 0.02^2) [n, k] on the GPU and quantize it to Q4_K there."""
    import synth
    w = scratch[: n * k]
    synth.normal_device(w, seed, tid, 0.02)
    out = torch.empty(n * k // 256 * 144, dtype=torch.uint8, device="cuda")
    fak.fak_q4k_pack_device(w, n, k, out)
    return out


def build_decode_model(fak, torch, n_layers=NL, vocab=V, seed=SEED_DECODE):
    """The 27B-shape stack: layer l % 4 == 3 is full-attention (q+gate, k, v, o), else GDN (in, out);
    every layer has gate/up/down; Q8_0 lm_head; f32 embedding.  Tensor ids 1000*l + slot."""
    import synth
    scratch = torch.empty(F * D, dtype=torch.float32, device="cuda")
    layers, q4_bytes = [], 0
    for l in range(n_layers):
        fa = l % 4 == 3
        L = {"kind": fak.FAK_LAYER_FA if fa else fak.FAK_LAYER_GDN}
        shapes = {"w_in": (0, QG if fa else GI, D), "w_out": (1, D, NM), "w_gate": (4, F, D), "w_up": (5, F, D),
                  "w_down": (6, D, F)}
        if fa:
            shapes.update({"w_k": (2, KV, D), "w_v": (3, KV, D)})
        for key, (slot, n, k) in shapes.items():
            L[key] = q4k_device(fak, torch, seed, 1000 * l + slot, n, k, scratch)
            q4_bytes += L[key].numel()
        layers.append(L)
    lm = torch.empty(vocab * D // 32 * 34, dtype=torch.uint8, device="cuda")
    rows = F * D // D  # chunk of lm_head rows that fits the scratch buffer
    for r0 in range(0, vocab, rows):
        nr = min(rows, vocab - r0)
        w = scratch[: nr * D]
        synth.normal_device(w, seed, 900000, 0.02, start=r0 * D)
        fak.fak_q8_0_pack_device(w, nr, D, lm[r0 * D // 32 * 34:(r0 + nr) * D // 32 * 34])
    emb = torch.empty(vocab * D, dtype=torch.float32, device="cuda")
    synth.normal_device(emb, seed, 900001, 1.0)
    del scratch
    torch.cuda.synchronize()
    return layers, lm, emb, q4_bytes + lm.numel()


def max_over_ranks(dist, torch, x, device):
    """The largest x over the ranks of the process group (x itself when there is no group): the job's
    time is its slowest replica's."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, ms):
    """Whole-job tokens/s of `world` independent replicas that each decode one token per `ms`."""
    return world * 1e3 / ms


def time_events(torch, fn, iters, warmup=3):
    """Average ms per call of fn() over `iters` after `warmup` untimed calls (lazy module loading, scratch pool
    growth), CUDA events on the current stream, synchronized both sides."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


# ------------------------------------------------------------------ headline: decode step
def bench_decode(fak, torch, args, dist, rank, world):
    layers, lm, emb, weight_bytes = build_decode_model(fak, torch, args.layers, args.vocab)
    ctx = fak.DecodeContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb, mode=fak.FAK_DECODE_ONE_LAUNCH)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(args.warmup):
        ctx.step(tok, tok)
    st = ctx.status()
    if st != 0:
        raise RuntimeError("decode warm-up status %d" % st)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            ctx.step(tok, tok)
        e1.record()
        torch.cuda.synchronize()
    ms = max_over_ranks(dist, torch, e0.elapsed_time(e1) / args.steps, "cuda")
    st = ctx.status()
    if st != 0:
        raise RuntimeError("decode status %d" % st)

    # end to end through the C ABI: the token goes host -> device before and device -> host after every step
    h_in = torch.zeros(1, dtype=torch.int32).pin_memory()
    h_out = torch.zeros(1, dtype=torch.int32).pin_memory()
    d_in = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_out = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_e2e = max(3, args.steps // 2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        d_in.copy_(h_in, non_blocking=True)
        ctx.step(d_in, d_out)
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.synchronize()
        h_in.copy_(h_out)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e

    # the same step launched once per matmul (the pages' per-command-buffer shape), for comparison
    ctx_pm = fak.DecodeContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb, mode=fak.FAK_DECODE_PER_MATMUL)
    for _ in range(2):
        ctx_pm.step(tok, tok)
    pm_ms = time_events(torch, lambda: ctx_pm.step(tok, tok), max(3, args.steps // 3))
    launches_pm = ctx_pm.launches_per_step()
    ctx_pm.close()
    # and with the host waiting for every launch before the next (the pages' commit-and-wait per
    # command buffer); the step returns only once the token has finished, so host time is exact
    ctx_hw = fak.DecodeContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb,
                               mode=fak.FAK_DECODE_PER_MATMUL_HOST_WAIT)
    ctx_hw.step(tok, tok)
    n_hw = 3
    t0 = time.perf_counter()
    for _ in range(n_hw):
        ctx_hw.step(tok, tok)
    hw_ms = (time.perf_counter() - t0) * 1e3 / n_hw
    ctx_hw.close()

    # the int8-activation variant of the same step (Q4_K steps on int8 x), and how far its logits
    # move from the exact step's on one token
    ctx_i8 = fak.DecodeContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb, mode=fak.FAK_DECODE_ONE_LAUNCH_I8X)
    i8_ms = time_events(torch, lambda: ctx_i8.step(tok, tok), max(3, args.steps // 3))
    t0_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    le, li = torch.empty(args.vocab, device="cuda"), torch.empty(args.vocab, device="cuda")
    o1, o2 = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.step(t0_tok, o1, le)
    ctx_i8.step(t0_tok, o2, li)
    st = ctx_i8.status()
    if st != 0:
        raise RuntimeError("int8 decode status %d" % st)
    le64, li64 = le.double(), li.double()
    i8_cos = float((le64 * li64).sum() / torch.sqrt((le64 * le64).sum() * (li64 * li64).sum()))
    i8_same_tok = int(o1.item()) == int(o2.item())
    ctx_i8.close()
    ctx.close()
    extra = {}
    if "mixer" in args.components:
        extra["decode_with_mixer"] = bench_decode_mixer(fak, torch, args, layers, lm, emb, weight_bytes)
    if "prefill_forward" in args.components:
        extra["prefill_forward"] = bench_prefill_forward(fak, torch, args, layers, lm, emb)
    del layers, lm, emb
    torch.cuda.empty_cache()
    algo_bytes = weight_bytes + D * 4  # + the embedding row read per token
    e2e_ms = max_over_ranks(dist, torch, e2e_ms, "cuda")
    return {"ms": ms, "tok_s": replica_throughput(world, ms), "clocks": clk.summary(), "algo_bytes": algo_bytes,
            "e2e_tok_s": replica_throughput(world, e2e_ms), "per_matmul_ms": pm_ms,
            "per_matmul_launches": launches_pm, "host_wait_ms": hw_ms, "i8x_ms": i8_ms, "i8x_logits_cosine": i8_cos,
            "i8x_same_token": i8_same_tok, "extra": extra}


def mixer_params_device(torch, n_layers, seed=SEED_DECODE):
    """Seeded mixer parameters per layer on the device (tensor ids 1000*l + 10..15): conv taps 0.5 N(0,1),
    a_log = log(1 + 15 u), dt_bias N(0,1), gated-norm and qk-norm gains 1 + 0.1 N(0,1)."""
    import numpy as np
    import synth
    conv_dim = 2 * MIX["gdn_nk"] * 128 + MIX["gdn_nv"] * 128
    out = []
    for l in range(n_layers):
        if l % 4 == 3:
            out.append({"q_norm_w": torch.from_numpy(1.0 + 0.1 * synth.normal(seed, 1000 * l + 14, (256,))).cuda(),
                        "k_norm_w": torch.from_numpy(1.0 + 0.1 * synth.normal(seed, 1000 * l + 15, (256,))).cuda()})
        else:
            u = synth.uniforms(seed, 1000 * l + 11, MIX["gdn_nv"])
            out.append({"conv_w": torch.from_numpy(0.5 * synth.normal(seed, 1000 * l + 10, (conv_dim, 4))).cuda(),
                        "a_log": torch.from_numpy(np.log(1.0 + 15.0 * u).astype(np.float32)).cuda(),
                        "dt_bias": torch.from_numpy(synth.normal(seed, 1000 * l + 12, (MIX["gdn_nv"],))).cuda(),
                        "norm_w": torch.from_numpy(1.0 + 0.1 * synth.normal(seed, 1000 * l + 13, (128,))).cuda()})
    return out


def bench_decode_mixer(fak, torch, args, layers, lm, emb, weight_bytes):
    """The same 64-layer step with the mixer bodies running on the GPU inside the launch: the Gated
    DeltaNet recurrence (conv state + 48 x 128 x 128 f32 state per GDN layer) and gated attention over
    a GPU-resident KV cache.  Timed over a sequence of `steps` positions from a reset."""
    mix = dict(MIX, max_ctx=4096, layers=mixer_params_device(torch, args.layers))
    ctx = fak.DecodeContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb, mode=fak.FAK_DECODE_ONE_LAUNCH,
                            mixer=mix)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(args.warmup):
        ctx.step(tok, tok)
    ctx.reset()
    n = max(3, args.steps)
    ms = time_events(torch, lambda: ctx.step(tok, tok), n, warmup=0)
    st = ctx.status()
    if st != 0:
        raise RuntimeError("mixer decode status %d" % st)
    ctx.close()
    n_gdn = sum(1 for l in range(args.layers) if l % 4 != 3)
    state_bytes = n_gdn * 2 * MIX["gdn_nv"] * 128 * 128 * 4  # S read and written per GDN layer
    return {"ms_per_step": ms, "tok_s": 1e3 / ms, "positions": n, "weights_bytes": weight_bytes,
            "gdn_state_bytes": state_bytes,
            "GBps": (weight_bytes + state_bytes) / (ms * 1e-3) / 1e9}


def bench_prefill_forward(fak, torch, args, layers, lm, emb):
    """The projections-only prefill forward of P tokens through the whole stack as one CUDA graph (the
    pages' prefill ladder, rung 3: both stage skips set), P = 256 / 512 / 1024."""
    out = []
    flops_tok = 0
    for l in range(args.layers):
        fa = l % 4 == 3
        flops_tok += 2 * D * ((QG + 2 * KV) if fa else GI) + 2 * NM * D + 2 * 2 * F * D + 2 * F * D
    for P in (256, 512, 1024):
        ctx = fak.PrefillContext(D, F, args.vocab, GI, QG, KV, NM, layers, lm, emb, P)
        toks = torch.arange(P, dtype=torch.int32, device="cuda") * 7919 % args.vocab
        tout = torch.zeros(1, dtype=torch.int32, device="cuda")
        ms = time_events(torch, lambda: ctx.run(toks, tout), 5, warmup=2)
        st = ctx.status()
        if st != 0:
            raise RuntimeError("prefill status %d" % st)
        out.append({"P": P, "ms": ms, "tok_s": P * 1e3 / ms, "TFLOPs": P * flops_tok / ms / 1e9,
                    "kernels_per_submission": ctx.kernels(), "submissions": 1})
        ctx.close()
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle baseline
_SAMPLE = {}


def cpu_oracle_sample(min_seconds=0.0):
    """Oracle throughput on this host: passes over one GDN layer (in_proj, out_proj, gate, up, down) and one
    full-attention layer (q+gate, k, v, o, gate, up, down) of the 27B stack (615 MB of Q4_K) plus 1/64 of
    the Q8_0 lm_head rows, dequantize + f64 dot, repeated until min_seconds of work (at least one pass).
    Returns (weight bytes per second, seconds, threads, description)."""
    import numpy as np
    import oracle
    import synth
    seed = SEED_DECODE
    if not _SAMPLE:  # inputs are built once; only the oracle's arithmetic is timed
        mats = []
        for l, shapes in ((0, ((0, GI, D), (1, D, NM), (4, F, D), (5, F, D), (6, D, F))),
                          (3, ((0, QG, D), (2, KV, D), (3, KV, D), (1, D, NM), (4, F, D), (5, F, D), (6, D, F)))):
            for slot, n, k in shapes:
                mats.append((oracle.q4k_pack(synth.normal(seed, 1000 * l + slot, (n, k), 0.02)), n, k, "q4"))
        nlm = V // 64
        mats.append((oracle.q8_0_pack(synth.normal(seed, 900000, (nlm, D), 0.02)), nlm, D, "q8"))
        _SAMPLE["mats"], _SAMPLE["x"] = mats, synth.normal(seed, 12345, (F,), 1.0)
    mats, x = _SAMPLE["mats"], _SAMPLE["x"]
    nbytes = sum(m[0].nbytes for m in mats)
    passes = 0
    t0 = time.perf_counter()
    while True:
        for W, n, k, kind in mats:
            (oracle.gemv_q4k if kind == "q4" else oracle.gemv_q8_0)(W, n, k, x[:k])
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    desc = "oracle (dequantize to f32, f64 dot), %d pass(es) in %.2f s over one GDN layer's 5 and one " \
           "full-attention layer's 7 Q4_K matrices + 1/64 of the Q8_0 lm_head (%.0f MB a pass), scaled to the " \
           "%.3f GB per token by bytes" % (passes, dt, nbytes / 1e6, 15.048048640)
    return passes * nbytes / dt, dt, threads, desc


def host_decode_model(n_layers=NL, vocab=V, seed=SEED_DECODE):
    """The 27B-shape stack on the host for the oracle: the same seeded weights as the device model, packed
    by the oracle's packer; the embedding table holds only the rows looked up (filled on demand)."""
    import numpy as np
    import oracle
    import synth
    layers = []
    for l in range(n_layers):
        fa = l % 4 == 3
        L = {"kind": oracle.LAYER_FA if fa else oracle.LAYER_GDN}
        shapes = {"w_in": (0, QG if fa else GI, D), "w_out": (1, D, NM), "w_gate": (4, F, D), "w_up": (5, F, D),
                  "w_down": (6, D, F)}
        if fa:
            shapes.update({"w_k": (2, KV, D), "w_v": (3, KV, D)})
        for key, (slot, n, k) in shapes.items():
            L[key] = oracle.q4k_pack(synth.normal(seed, 1000 * l + slot, (n, k), 0.02))
        layers.append(L)
    rows = 8192
    lm = np.concatenate([oracle.q8_0_pack(synth.normal(seed, 900000, (min(rows, vocab - r0), D), 0.02,
                                                       start=r0 * D)).reshape(-1) for r0 in range(0, vocab, rows)])
    emb = np.zeros((vocab, D), np.float32)  # untouched pages cost no memory
    model = oracle.Model(D, F, vocab, GI, QG, KV, NM, layers, lm, emb)

    def need_row(t):
        emb[t] = synth.normal(seed, 900001, (D,), 1.0, start=t * D)
    return model, need_row


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, each step one whole decode token of the 27B-shape stack
    (all 64 layers and the lm_head, 15.05 GB of Q4_K / Q8_0 weights), free-running from token 0 as the GPU
    step is; timed on this host's cores.  The host model is built first, outside the timed steps."""
    if rank != 0:
        return
    model, need_row = host_decode_model(args.layers, args.vocab)
    full = args.layers == NL and args.vocab == V
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    tok, secs = 0, []
    for i in range(args.warmup + args.steps):
        need_row(tok)
        t0 = time.perf_counter()
        tok = model.decode_token(tok)[0]
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            secs.append(dt)
    ms = 1e3 * statistics.mean(secs)
    v = 1e3 / ms
    desc = "oracle (dequantize to f32, f64 dot), %d whole %d-layer tokens timed one by one (after %d untimed), " \
           "%.3f GB of weights each" % (args.steps, args.layers, args.warmup, model.weight_bytes() / 1e9)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "27B-shape hybrid decode step, batch 1, whole tokens" if full else
                   "REDUCED profiling case of the 27B-shape decode step: %d layers, Q8_0 lm_head 5120->%d "
                   "(not the headline)" % (args.layers, args.vocab)},
        "cpu_baseline": {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ------------------------------------------------------------------ components
def graph_time(torch, fn, reps, iters=5):
    """Device time per call of fn() (us) with host launch cost removed: `reps` calls captured in one CUDA
    graph, replayed `iters` times, CUDA events on the replaying stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (iters * reps) * 1e3


def bench_components(fak, torch, hbm, bf16, which):
    """Component sections.  GEMV-like calls are timed two ways: 'us' = device time per call back to back
    (CUDA graph of many calls on rotating weight copies totalling > 4 x L2, so every call reads W from HBM),
    'us_eager' = the same through the Python binding launch by launch (includes host launch cost)."""
    import synth
    out = {}

    def rotating(W, copies):
        return [W] + [W.clone() for _ in range(copies - 1)]

    if "gemv" in which:
        def gemv_case(N, K, seed, wid, xid):
            copies = max(1, min(60, int(600e6 // (N * K * 0.5625))))
            scratch = torch.empty(N * K, dtype=torch.float32, device="cuda")
            Ws = rotating(q4k_device(fak, torch, seed, wid, N, K, scratch), copies)
            del scratch
            x = torch.empty(K, device="cuda")
            synth.normal_device(x, seed, xid, 1.0)
            y = torch.empty(N, device="cuda")
            it = [0]

            def one():
                fak.fak_q4k_gemv(Ws[it[0] % copies], N, K, x, y)
                it[0] += 1

            def one_i8():
                fak.fak_q4k_gemv_i8x(Ws[it[0] % copies], N, K, x, y)
                it[0] += 1
            reps = max(copies, 20) if copies > 1 else 5
            us = graph_time(torch, one, reps)
            ue = time_events(torch, one, 50 if N * K < 100_000_000 else 10) * 1e3
            us8 = graph_time(torch, one_i8, reps)
            byts = N * K // 256 * 144 + 4 * (N + K)
            return {"N": N, "K": K, "us": us, "GBps": byts / us / 1e3, "frac": byts / us / 1e3 / hbm,
                    "us_eager": ue, "rotating_copies": copies, "bytes": byts,
                    "int8_activations": {"us": us8, "GBps": byts / us8 / 1e3, "frac": byts / us8 / 1e3 / hbm}}

        # single GEMV 5120 x 5120 (seed 0: W tensor 0, x tensor 1)
        out["gemv_5120x5120"] = gemv_case(5120, 5120, 0, 0, 1)
        # GEMV shape sweep (seed 4: W shape i -> tensor i, x -> 100 + i)
        out["gemv_sweep"] = [gemv_case(N, K, 4, i, 100 + i) for i, (N, K) in
                             enumerate([(1024, 5120), (5120, 5120), (17408, 5120), (5120, 17408), (248320, 5120)])]

    if "mlp" in which or "batch" in which:
        # batch-1 MLP weights (seed 1: x 0, gate 1, up 2, down 3), 4 rotating copies = 601 MB
        scratch = torch.empty(F * D, dtype=torch.float32, device="cuda")
        g = q4k_device(fak, torch, 1, 1, F, D, scratch)
        u = q4k_device(fak, torch, 1, 2, F, D, scratch)
        dn = q4k_device(fak, torch, 1, 3, D, F, scratch)
        del scratch
        mlps = [(g, u, dn)] + [(g.clone(), u.clone(), dn.clone()) for _ in range(3)]
        it = [0]
        if "mlp" in which:
            x = torch.empty(D, device="cuda")
            synth.normal_device(x, 1, 0, 1.0)
            y = torch.empty(D, device="cuda")
            ws = torch.empty(fak.fak_mlp_workspace_bytes(F), dtype=torch.uint8, device="cuda")

            def mlp():
                a, b, c = mlps[it[0] % 4]
                fak.fak_mlp_decode(a, b, c, D, F, x, 1e-6, y, ws)
                it[0] += 1
            us = graph_time(torch, mlp, 20)
            ue = time_events(torch, mlp, 100) * 1e3
            mb = 3 * F * D // 256 * 144 + 4 * (2 * D + F)
            out["mlp_decode"] = {"us": us, "GBps": mb / us / 1e3, "frac": mb / us / 1e3 / hbm, "us_eager": ue,
                                 "bytes": mb, "launches_per_call": 1}
        if "batch" in which:
            # batched GEMV sweep on the gate weight (seed 1, X tensor 4 rows 0..M-1)
            Xall = torch.empty(64 * D, device="cuda")
            synth.normal_device(Xall, 1, 4, 1.0)
            bs = []
            for M in (1, 2, 4, 8, 16, 32, 64):
                Y = torch.empty(M * F, device="cuda")

                def bat():
                    fak.fak_q4k_gemv_batch(mlps[it[0] % 4][0], F, D, Xall, M, Y)
                    it[0] += 1
                us = graph_time(torch, bat, 20)
                ue = time_events(torch, bat, 20) * 1e3
                byts = F * D // 256 * 144 + 4 * M * (D + F)
                bs.append({"M": M, "us": us, "GBps": byts / us / 1e3, "frac": byts / us / 1e3 / hbm,
                           "GFLOPs": 2.0 * M * F * D / us / 1e3, "us_per_row": us / M, "us_eager": ue})
            out["gemv_batch_sweep"] = bs
        del mlps, g, u, dn

    if "prefill" in which:
        # prefill GEMMs (seed 2: W1 gate||up tensor 0, W2 down tensor 1, X tensor 2)
        scratch = torch.empty(2 * F * D, dtype=torch.float32, device="cuda")
        W1 = q4k_device(fak, torch, 2, 0, 2 * F, D, scratch)
        W2 = q4k_device(fak, torch, 2, 1, D, F, scratch)
        Xf = scratch[: 1024 * D]
        synth.normal_device(Xf, 2, 2, 1.0)
        X = Xf.view(1024, D).to(torch.bfloat16)
        del scratch, Xf
        row = D // 256 * 144
        W13 = torch.empty_like(W1)  # gate / up rows interleaved by 16 for the fused SwiGLU epilogue
        fak.fak_q4k_interleave_gate_up(W1[: F * row], W1[F * row:], F, D, W13)
        pre = []
        for P in (256, 512, 1024):
            Y1 = torch.empty(P * 2 * F, device="cuda")
            X2 = torch.empty(P * F, dtype=torch.bfloat16, device="cuda")
            Y2 = torch.empty(P * D, device="cuda")
            m1 = time_events(torch, lambda: fak.fak_q4k_gemm(W1, 2 * F, D, X, P, Y1), 10)
            ms_sw = time_events(torch, lambda: fak.fak_swiglu_bf16(Y1, P, F, X2), 10)
            m2 = time_events(torch, lambda: fak.fak_q4k_gemm(W2, D, F, X2, P, Y2), 10)
            mf = time_events(torch, lambda: fak.fak_q4k_gemm_swiglu(W13, F, D, X, P, X2), 10)
            f1, f2 = 2.0 * P * 2 * F * D, 2.0 * P * D * F
            pre.append({"P": P, "gate_up_ms": m1, "gate_up_TFLOPs": f1 / m1 / 1e9,
                        "gate_up_frac": f1 / m1 / 1e9 / bf16, "swiglu_ms": ms_sw, "down_ms": m2,
                        "down_TFLOPs": f2 / m2 / 1e9, "down_frac": f2 / m2 / 1e9 / bf16,
                        "total_TFLOPs": (f1 + f2) / (m1 + ms_sw + m2) / 1e9,
                        "gate_up_swiglu_fused_ms": mf, "gate_up_swiglu_fused_TFLOPs": f1 / mf / 1e9,
                        "total_fused_TFLOPs": (f1 + f2) / (mf + m2) / 1e9})
        out["prefill_gemm"] = pre
    st = fak.fak_device_status()
    if st != 0:
        raise RuntimeError("component status %d" % st)
    return out


# dram bytes (read + write) of one full decode launch: the ncu capture of the same engine kernel on the
# 4-layer stack (955.81 MB for 945.22 MB of weights), scaled by weight bytes to the 15.048 GB step.
# Set to None whenever the engine kernel changes until re-captured.
DECODE_TRAFFIC_BYTES = int(955.814144e6 / 945.22368e6 * (15_048_048_640 + 5120 * 4))


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import __graft_entry__
    __graft_entry__.build()
    import torch
    import q4_weight_quantized_block_gb300 as fak
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    dec = bench_decode(fak, torch, args, dist, rank, world)
    comps = None
    if rank == 0 and args.components:
        comps = bench_components(fak, torch, hbm, bf16, args.components)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        bps, dt, threads, desc = cpu_oracle_sample(10.0)
        cpu = {"value": bps / dec["algo_bytes"], "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": desc,
               "sample_seconds": dt}
    if dist:
        dist.barrier()
    if rank != 0:
        return
    achieved = dec["algo_bytes"] / (dec["ms"] * 1e-3) / 1e9
    full = args.layers == NL and args.vocab == V
    workload = ("27B-shape hybrid decode step, batch 1: 64 layers (48 GDN: in 5120->16480, out 6144->5120; 16 FA: "
                "q+gate 5120->12288, k/v 5120->1024, o 6144->5120; MLP 5120->2x17408->5120), RMSNorm, SwiGLU, "
                "Q8_0 lm_head 5120->248320 + argmax") if full else (
        "REDUCED profiling case of the 27B-shape decode step: %d layers, Q8_0 lm_head 5120->%d (not the headline)"
        % (args.layers, args.vocab))
    line = {
        "metric": METRIC, "value": dec["tok_s"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dec["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded N(0,0.02^2) weights quantized to Q4_K / Q8_0 on the GPU, N(0,1) embedding",
        "config": {"workload": workload,
                   "weights_bytes_per_token": dec["algo_bytes"], "launch": "one kernel per token",
                   "l2": "weights per token %.2f GB >> L2 129 MB: no flush needed" % (dec["algo_bytes"] / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": DECODE_TRAFFIC_BYTES if full else None, "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "engine_kernel (one-launch decode step)"},
        "cpu_baseline": cpu,
        "e2e": {"value": dec["e2e_tok_s"], "unit": "tok/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4},
        "clocks": dec["clocks"],
        "gpu_launches": args.steps,
        "per_matmul_mode": {"ms_per_step": dec["per_matmul_ms"], "tok_s": 1e3 / dec["per_matmul_ms"],
                            "launches_per_step": dec["per_matmul_launches"]},
        "per_matmul_host_wait_mode": {"ms_per_step": dec["host_wait_ms"], "tok_s": 1e3 / dec["host_wait_ms"],
                                      "launches_per_step": dec["per_matmul_launches"],
                                      "timing": "host clock over 3 steps; every launch waited on"},
        "decode_with_mixer": dec["extra"].get("decode_with_mixer"),
        "prefill_forward": dec["extra"].get("prefill_forward"),
        "int8_activation_variant": {"ms_per_step": dec["i8x_ms"], "tok_s": 1e3 / dec["i8x_ms"],
                                    "roofline_frac": dec["algo_bytes"] / (dec["i8x_ms"] * 1e-3) / 1e9 / hbm,
                                    "logits_cosine_vs_exact": dec["i8x_logits_cosine"],
                                    "same_token_as_exact": dec["i8x_same_token"]},
        "components": comps,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
