"""Benchmark of the MoE FFN layer on GB300 (one JSON line on rank 0).

Workload (synthetic, seeded; shapes of the MoE layer in "Optimizing on-device inference for
Apple Silicon": 256 experts, top 8 plus a shared expert, 4K-token prompts, batch-1 decode):
  step = one layer forward at T=4096 tokens, d=2048, expert inner dim 512, balanced routing
  (x ~ N(0,1), router ~ N(0,0.05), experts ~ N(0,0.02)), through moe_forward on device
  buffers.  value = tokens/s over all ranks (each rank runs its own batch: weak scaling).
Also measured in the same run and reported in the same line:
  decode: batch-1 (T=1) over 40 independent layers' weights (64.7 GB, defeats L2), one CUDA
          graph of 40 stream-ordered layer calls; us/layer and HBM GB/s;
  roofline: the dominant kernel of the step, algorithmic bytes (or FLOPs) per launch over
          its CUDA-event duration, against MEASURED_PEAKS.json;
  e2e: the same tokens/s through moe_forward_host (pinned host x in, host y out, copies
       inside the timed region);
  cpu_baseline: the CPU oracle on a bounded sample of the same workload (rank 0 only);
  prefill_skewed: the same layer with skewed routing (router bias -2.4 ln(rank_e)), timed
       and set against the floor of its own bytes and FLOPs;
  prefill_sweep: the balanced layer at T = 256 .. 131072 (bf16; --sweep-q4 adds 4-bit experts),
       each T with the floor of its bytes and FLOPs;
  gdn_scan: the Gated DeltaNet recurrent scan of one layer (32 heads, 128 x 128 fp32 state)
       over 2K- and 16K-token prompts, us per scan against the SMs' fp32 FMA peak, with the
       scan oracle's rate on the host cores.
--impl reference times only the CPU oracle (the reference arm of this benchmark).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer prefill tokens/s @T=4096 & decode us/layer (T=1); % of roofline"
T_PREFILL, D, F, FS, E, K = 4096, 2048, 512, 512, 256, 8
DECODE_LAYERS = 40
FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2
KERNELS_GEMM = ("router_topk", "route_plan_scatter", "experts", "combine")
KERNELS_GEMV = ("decode_router_shared", "decode_gateup", "decode_down_combine")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target duration of the CPU oracle sample")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="decode only (profiling runs)")
    p.add_argument("--decode-layers", type=int, default=DECODE_LAYERS,
                   help="layers in the decode graph (40 = the benchmark workload)")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-skew", action="store_true", help="skip the skewed-routing prefill line")
    p.add_argument("--no-q4", action="store_true", help="skip the 4-bit prefill and decode lines")
    p.add_argument("--no-small-batch", action="store_true",
                   help="skip the T = 2..5 decode lines")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the prefill length sweep (T = 256 .. 131072, balanced, bf16)")
    p.add_argument("--sweep-q4", action="store_true",
                   help="also run the length sweep with 4-bit experts")
    p.add_argument("--sweep-tokens", type=str, default=None,
                   help="comma-separated T values of the sweep (default: 256 .. 131072)")
    p.add_argument("--no-gdn", action="store_true",
                   help="skip the Gated DeltaNet scan line (T = 2048, 32 heads of 128 x 128)")
    p.add_argument("--gdn-tokens", type=str, default="2048,16384",
                   help="comma-separated prompt lengths of the Gated DeltaNet scan line")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        P = json.load(open(path))
        return float(P["hbm_gbs"]), float(P["bf16_tflops"]), "of measured"
    except Exception:
        return 6800.0, 1900.0, "of fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- workload bytes and flops

def algorithmic(counts, T):
    """Algorithmic bytes and FLOPs of one prefill layer and of its kernels: weights of the
    non-empty experts, the shared expert and the router, x in and y out; FLOPs of the GEMMs
    actually needed (8 routed + 1 shared per token, router)."""
    ne = int((counts > 0).sum())
    S = T * K
    b = dict(
        router_topk=E * D * 2 + T * D * 2,
        experts=ne * 3 * F * D * 2 + 3 * FS * D * 2 + T * D * 2,  # weights + x
        combine=T * D * 2,
    )
    fl = dict(
        router_topk=2 * T * E * D,
        experts=2 * (S * 3 * F + T * 3 * FS) * D,
    )
    layer_bytes = E * D * 2 + ne * 3 * F * D * 2 + 3 * FS * D * 2 + 2 * T * D * 2
    layer_flops = fl["router_topk"] + fl["experts"]
    return b, fl, layer_bytes, layer_flops


DECODE_BYTES_PER_LAYER = 9 * 3 * F * D * 2 + E * D * 2 + 2 * D * 2  # 9 experts + router + x + y
# 4-bit experts: half a byte per weight plus a bf16 scale and bias per 64; the router stays bf16
DECODE_Q4_BYTES_PER_LAYER = 9 * 3 * F * D * 9 // 16 + E * D * 2 + 2 * D * 2  # 0.5625 B/weight


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_smi_id(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else dev


# ---------------------------------------------------------------- CPU oracle

def oracle_sample_rate(target_s, threads=None):
    """tokens/s of the CPU oracle on a sample of the T=4096 prefill workload, sized to take
    about target_s seconds; returns (rate, sample description, cores)."""
    import oracle
    dims = synth.Dims(d=D, f=F, fs=FS)
    x = synth.x_rows(0, 0, T_PREFILL, D)
    w_r = synth.host_weight(0, 0, "w_r", dims)
    W = {n: synth.host_weight(0, 0, n, dims) for n in synth.WEIGHT_NAMES if n != "w_r"}
    experts = (W["w_gate"], W["w_up"], W["w_down"])
    shared = (W["ws_gate"], W["ws_up"], W["ws_down"])
    cores = threads or host_cores()
    n = max(1, cores)
    toks = np.arange(n) * (T_PREFILL // n)
    t0 = time.perf_counter()
    oracle.forward(x, w_r, None, experts, shared, K, tokens=toks, nthreads=cores)
    dt = time.perf_counter() - t0
    n2 = int(min(T_PREFILL, max(n, n * target_s / max(dt, 1e-3))))
    n2 = max(cores, n2 // cores * cores)
    toks = np.linspace(0, T_PREFILL - 1, n2).astype(np.int64)
    t0 = time.perf_counter()
    oracle.forward(x, w_r, None, experts, shared, K, tokens=toks, nthreads=cores)
    dt = time.perf_counter() - t0
    return n2 / dt, f"{n2} of the 4096 prefill tokens (evenly spaced), full layer per token", cores


def reference_arm(args, rank):
    if rank != 0:
        return
    import oracle
    dims = synth.Dims(d=D, f=F, fs=FS)
    x = synth.x_rows(0, 0, T_PREFILL, D)
    w_r = synth.host_weight(0, 0, "w_r", dims)
    W = {n: synth.host_weight(0, 0, n, dims) for n in synth.WEIGHT_NAMES if n != "w_r"}
    experts = (W["w_gate"], W["w_up"], W["w_down"])
    shared = (W["ws_gate"], W["ws_up"], W["ws_down"])
    cores = host_cores()
    # one step = the oracle on `n` tokens; n sized so that all steps fit in about 2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = cores
    t0 = time.perf_counter()
    oracle.forward(x, w_r, None, experts, shared, K, tokens=np.arange(n), nthreads=cores)
    per_tok = (time.perf_counter() - t0) / n
    n = int(max(cores, min(T_PREFILL, budget / max(per_tok, 1e-6) // cores * cores)))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.forward(x, w_r, None, experts, shared, K,
                       tokens=rng.choice(T_PREFILL, n, replace=False), nthreads=cores)
    times = []
    for _ in range(args.steps):
        toks = rng.choice(T_PREFILL, n, replace=False)
        t0 = time.perf_counter()
        oracle.forward(x, w_r, None, experts, shared, K, tokens=toks, nthreads=cores)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n / (ms / 1e3)
    sample = f"{n} random tokens of the T=4096 prefill workload per step, full layer per token"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "prefill T=4096 d=2048 E=256 top-8 f=512 + shared (balanced)",
                   "T": T_PREFILL, "d": D, "experts": E, "top_k": K, "ffn_dim": F,
                   "shared_ffn_dim": FS},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def device_weights(torch, seed, layer, dims, bias=None):
    W = {}
    s = torch.cuda.current_stream().cuda_stream
    for nm in synth.WEIGHT_NAMES:
        t = torch.empty(synth.weight_shape(nm, dims), dtype=torch.bfloat16, device="cuda")
        synth.device_weight(seed, layer, nm, dims, t.data_ptr(), s)
        W["w_router" if nm == "w_r" else nm] = t
    if bias is not None:
        W["router_bias"] = torch.from_numpy(bias).cuda()
    return W


def run_prefill(torch, moe, args, rank, world, P_hbm, P_tc, peak_note):
    dims = synth.Dims(d=D, f=F, fs=FS)
    seed = rank  # each rank its own batch and weights
    W = device_weights(torch, seed, 0, dims)
    x = torch.from_numpy(synth.x_rows(seed, 0, T_PREFILL, D).view(np.int16)).cuda() \
        .view(torch.bfloat16)
    y = torch.empty_like(x)
    layer = moe.MoeLayer(W, T_PREFILL)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    counts = np.diff(layer.route(x)["offsets"].cpu().numpy())
    for _ in range(args.warmup):
        layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.device_error() == moe.MOE_OK

    # headline: per-step device time of the layer, L2 flushed (untimed) before each step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for a, b in ev:
        flush.zero_()
        a.record()
        layer.forward(x, y)
        b.record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = reduce_max(torch, world, statistics.mean(step_ms))

    # per-kernel durations (events between the kernels; kernels serialised)
    nprof = min(args.steps, 200)
    assert moe.moe_profile_begin(layer.handle, nprof) == moe.MOE_OK
    for _ in range(nprof):
        flush.zero_()
        layer.forward(x, y)
    st, kms, ncalls = moe.moe_profile_end(layer.handle)
    assert st == moe.MOE_OK and ncalls == nprof
    kms = [t / ncalls for t in kms]

    # end to end through the host entry point
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        layer.forward_host(xh, yh)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in ev2:
        flush.zero_()
        a.record()
        layer.forward_host(xh, yh)
        b.record()
    torch.cuda.synchronize()
    e2e_ms = reduce_max(torch, world, statistics.mean(a.elapsed_time(b) for a, b in ev2))
    assert layer.device_error() == moe.MOE_OK

    byts, flops, layer_bytes, layer_flops = algorithmic(counts, T_PREFILL)
    kt = dict(zip(KERNELS_GEMM, kms))
    dom = max(kt, key=kt.get)
    t_dom = kt[dom] / 1e3
    ridge = P_tc * 1e12 / (P_hbm * 1e9)
    if dom in flops and flops[dom] / byts[dom] > ridge:
        roof = {"bound": "tensor", "achieved": flops[dom] / t_dom / 1e12, "peak": P_tc,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": byts[dom] / t_dom / 1e9, "peak": P_hbm,
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["peak_source"] = peak_note
    roof["traffic"] = profiled_traffic(dom)
    roof["kernel_ms"] = {k: round(v, 5) for k, v in kt.items()}
    t_layer = ms / 1e3
    stats = {"hbm_frac": layer_bytes / t_layer / 1e9 / P_hbm,
             "tensor_frac": layer_flops / t_layer / 1e12 / P_tc,
             "algorithmic_bytes": layer_bytes, "flops": layer_flops,
             "nonempty_experts": int((counts > 0).sum()), "timed_wall_s": t_wall}
    layer.close()
    return dict(ms=ms, e2e_ms=e2e_ms, roofline=roof, layer=stats, launches=len(KERNELS_GEMM))


SWEEP_T = (256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)


def time_prefill(torch, moe, T, skew, steps, warmup, seed, P_hbm, P_tc, q4=False):
    """Layer time (L2 flushed before every step) at T tokens, balanced or skewed routing
    (router bias -2.4 ln(rank) over a seeded permutation of the experts), with the bytes and
    FLOPs of that routing and the fraction of the binding floor max(bytes/B, FLOPs/P).  With
    q4 the experts are 4-bit (4.5 bits per weight with the group scales and biases)."""
    dims = synth.Dims(d=D, f=F, fs=FS)
    bias = synth.skew_bias(seed, 0, E) if skew else None
    W = (q4_device_weights if q4 else device_weights)(torch, seed, 0, dims, bias)
    x = torch.from_numpy(synth.x_rows(seed, 0, T, D).view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    layer = moe.MoeLayer(W, T)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    counts = np.diff(layer.route(x)["offsets"].cpu().numpy())
    for _ in range(warmup):
        layer.forward(x, y)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record()
        layer.forward(x, y)
        b.record()
    torch.cuda.synchronize()
    assert layer.device_error() == moe.MOE_OK
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    layer.close()
    _, _, byts, flops = algorithmic(counts, T)
    if q4:
        ne = int((counts > 0).sum())
        byts -= (ne * 3 * F * D + 3 * FS * D) * 23 // 16  # 2 bytes -> 9/16 byte per weight
    t = ms / 1e3
    floor = max(byts / (P_hbm * 1e9), flops / (P_tc * 1e12))
    return {"T": T, "routing": "skewed" if skew else "balanced", "weights": "4-bit" if q4 else
            "bf16", "ms": ms,
            "tokens_per_s": T / t, "hbm_frac": byts / t / 1e9 / P_hbm,
            "tensor_frac": flops / t / 1e12 / P_tc, "floor_us": floor * 1e6,
            "frac_of_floor": floor / t, "bound": "hbm" if byts / (P_hbm * 1e9) >= flops /
            (P_tc * 1e12) else "tensor", "nonempty_experts": int((counts > 0).sum()),
            "max_expert_rows": int(counts.max())}


# ---------------------------------------------------------------- Gated DeltaNet scan

GDN_H, GDN_DK, GDN_DV = 32, 128, 128
SM_CLOCK_MHZ = 2070.0  # GB300's maximum SM clock (the clock samples of the run are reported)


def gdn_algorithmic(T, H=GDN_H, dk=GDN_DK, dv=GDN_DV):
    """FLOPs and bytes of one scan as the rule is written: per token and head S^T k (2 dk dv),
    the delta u (3 dv), alpha S + k u^T (3 dk dv), S^T q (2 dk dv); bytes: q, k, v, o in bf16,
    the gates in fp32, the state read and written once in fp32."""
    flops = T * H * (7 * dk * dv + 3 * dv)
    byts = T * H * (2 * dk * 2 + 2 * dv * 2 + 2 * 4) + 2 * H * dk * dv * 4
    return flops, byts


def run_gdn(torch, moe, args, P_hbm, rank=0, world=1):
    """The Gated DeltaNet recurrent scan of one layer (32 heads, 128 x 128 fp32 state each)
    over a prompt of T tokens: device time per scan (L2 flushed before every step), against
    the fp32 FMA peak of the SMs (the scan is FMA-bound: 4 FMA-pipe operations per state
    element and token), with the oracle's rate on the host cores beside it."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    peak_tf = sms * 128 * 2 * SM_CLOCK_MHZ * 1e6 / 1e12
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    rows = []
    for T in [int(t) for t in args.gdn_tokens.split(",") if t]:
        H, dk, dv = GDN_H, GDN_DK, GDN_DV
        q = torch.empty((T, H, dk), dtype=torch.int16, device="cuda")
        k = torch.empty_like(q)
        v = torch.empty((T, H, dv), dtype=torch.int16, device="cuda")
        al = torch.empty((T, H), dtype=torch.float32, device="cuda")
        be = torch.empty_like(al)
        s0b = torch.empty((H, dk, dv), dtype=torch.int16, device="cuda")
        synth.gdn_inputs_device(0, T, H, dk, dv, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                al.data_ptr(), be.data_ptr(), s0b.data_ptr(),
                                cuda_stream=stream.cuda_stream)
        s0 = s0b.view(torch.bfloat16).float()  # exact widening of the bf16 draws
        s1 = torch.empty_like(s0)
        o = torch.empty((T, H, dv), dtype=torch.int16, device="cuda")

        def scan():
            st = moe.gdn_scan(q.data_ptr(), k.data_ptr(), v.data_ptr(), al.data_ptr(),
                              be.data_ptr(), s0.data_ptr(), s1.data_ptr(), o.data_ptr(), T, H,
                              dk, dv, stream.cuda_stream)
            assert st == moe.MOE_OK, moe.moe_status_string(st)

        for _ in range(max(3, args.warmup)):
            scan()
        steps = min(args.steps, 50)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            scan()
            b.record(stream)
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
        flops, byts = gdn_algorithmic(T)
        tf = flops / (us * 1e-6) / 1e12
        rows.append({
            "T": T, "heads": H, "dk": dk, "dv": dv, "us": us, "tokens_per_s": T / (us * 1e-6),
            "roofline": {"bound": "alu", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": tf / peak_tf,
                         "peak_source": f"derived: {sms} SMs x 128 fp32 lanes x 2 FLOP x "
                                        f"{SM_CLOCK_MHZ:.0f} MHz",
                         # DRAM bytes of one launch from the committed capture (taken at
                         # T = 2048 on this kernel source), for that row only
                         "traffic": profiled_traffic("gdn_scan") if T == 2048 else None},
            "hbm_frac": byts / (us * 1e-6) / 1e9 / P_hbm,
            "algorithmic_flops": flops, "algorithmic_bytes": byts, "gpu_launches": steps,
            "l2": "flushed (256 MB write, untimed) before every timed step"})
        del q, k, v, al, be, s0b, s0, s1, o
    # the oracle's rate on the host cores: rank 0 of a one-GPU run only
    cpu = None if args.no_cpu or rank != 0 or world != 1 else gdn_oracle_rate()
    return {"rows": rows, "cpu_baseline": cpu}


def gdn_oracle_rate(T=2048):
    """The scan oracle (fp64, one head per host thread) on the T=2048, 32-head layer."""
    import time

    import oracle
    q, k, v, al, be, s0 = synth.gdn_inputs(0, T, GDN_H, GDN_DK, GDN_DV)
    cores = host_cores()
    t0 = time.perf_counter()
    oracle.gdn_scan(q, k, v, al, be, s0, nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": T / dt, "unit": "tokens/s", "cores": min(cores, GDN_H), "kind": "oracle",
            "sample": f"the whole T={T}, {GDN_H}-head scan, one head per thread"}


def run_decode(torch, moe, args, rank, world, P_hbm):
    dims = synth.Dims(d=D, f=F, fs=FS)
    seed = 1000 + rank
    layers, Ws = [], []
    nl = args.decode_layers
    for l in range(nl):
        W = device_weights(torch, seed, l, dims)
        Ws.append(W)
        layers.append(moe.MoeLayer(W, 1, schedule=moe.MOE_SCHEDULE_GEMV))
    x = torch.from_numpy(synth.x_rows(seed, 0, 1, D).view(np.int16)).cuda().view(torch.bfloat16)
    ys = [torch.empty_like(x) for _ in range(nl)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for L, y in zip(layers, ys):  # eager warm-up before capture
            L.forward(x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for L, y in zip(layers, ys):
            L.forward(x, y)
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(torch, world, statistics.median(a.elapsed_time(b) for a, b in ev))
    us_layer = ms * 1e3 / nl
    gbs = DECODE_BYTES_PER_LAYER / (us_layer * 1e-6) / 1e9
    # per-kernel split of one layer (eager, serialised)
    L0 = layers[0]
    assert moe.moe_profile_begin(L0.handle, 50) == moe.MOE_OK
    for _ in range(50):
        L0.forward(x, ys[0])
    st, kms, nc = moe.moe_profile_end(L0.handle)
    for L in layers:
        assert L.device_error() == moe.MOE_OK
        L.close()
    read_gbs = read_probe(torch, moe)
    small = None if args.no_small_batch else run_small_batch(torch, moe, args, Ws, seed, P_hbm)
    del Ws
    q4 = None if args.no_q4 else run_decode_q4(torch, moe, args, seed, P_hbm)
    return {"us_per_layer": us_layer, "GB_per_s": gbs, "layers": nl,
            "bytes_per_layer": DECODE_BYTES_PER_LAYER,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": P_hbm, "unit": "GB/s",
                         "frac": gbs / P_hbm},
            "kernel_us_eager": decode_kernel_times(kms, nc),
            "read_probe": {"GB_per_s": read_gbs, "frac_of_read_probe": gbs / read_gbs,
                           "how": "moe_read_probe over 4 GiB, best of 10 (a read-only stream; "
                                  "the roofline peak above stays the measured copy rate)"},
            "gpu_launches": args.steps * nl * 3,
            "graph": f"{nl} stream-ordered layer calls, replayed per step",
            "small_batch": small,
            "q4": q4}


def decode_kernel_times(kms, nc):
    """Per-kernel eager times (us) of one batch-1 layer from moe_profile_end: the router
    launch, then either the streamed launch (its second slot empty) or the gate/up and the
    down+combine launches."""
    us = [v / nc * 1e3 for v in kms]
    # the two-launch form's down+combine kernel takes about as long as its gate/up kernel; an
    # empty slot is a small fraction of the streamed launch
    if len(us) == 3 and us[2] < 0.3 * us[1]:
        # the third slot holds no kernel: eager launches leave the GPU waiting on the host
        # between two events, which is all that slot measures
        return {"decode_router": round(us[0], 3), "decode_expert_stream": round(us[1], 3),
                "empty_slot_host_gap": round(us[2], 3)}
    return {k: round(v, 3) for k, v in zip(KERNELS_GEMV, us)}


def q4_device_weights(torch, seed, layer, dims, bias=None):
    """Device 4-bit experts (codes, scales, biases per tensor) and the bf16 router."""
    s = torch.cuda.current_stream().cuda_stream
    W = {"w_router": torch.empty((E, dims.d), dtype=torch.bfloat16, device="cuda")}
    synth.device_weight(seed, layer, "w_r", dims, W["w_router"].data_ptr(), s)
    for nm in synth.Q4_NAMES:
        cs, gs = synth.q4_shapes(nm, dims)
        t = (torch.empty(cs, dtype=torch.uint8, device="cuda"),
             torch.empty(gs, dtype=torch.bfloat16, device="cuda"),
             torch.empty(gs, dtype=torch.bfloat16, device="cuda"))
        synth.q4_device(seed, layer, nm, dims, *(a.data_ptr() for a in t), s)
        W[nm] = t
    if bias is not None:
        W["router_bias"] = torch.from_numpy(bias).cuda()
    return W


def run_prefill_q4(torch, moe, args, seed, P_hbm, P_tc):
    """Prefill T=4096 (balanced routing) with 4-bit experts on the tensor-core path: the
    grouped GEMM dequantizes each weight tile into tensor memory.  Layer time with L2 flushed
    before each step, the per-kernel split, and the expert kernel against the bf16 tensor
    peak (its FLOPs are those of the bf16 layer)."""
    dims = synth.Dims(d=D, f=F, fs=FS)
    W = q4_device_weights(torch, seed, 0, dims)
    x = torch.from_numpy(synth.x_rows(seed, 0, T_PREFILL, D).view(np.int16)).cuda() \
        .view(torch.bfloat16)
    y = torch.empty_like(x)
    layer = moe.MoeLayer(W, T_PREFILL)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    counts = np.diff(layer.route(x)["offsets"].cpu().numpy())
    for _ in range(max(3, args.warmup)):
        layer.forward(x, y)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record()
        layer.forward(x, y)
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nprof = min(args.steps, 50)
    assert moe.moe_profile_begin(layer.handle, nprof) == moe.MOE_OK
    for _ in range(nprof):
        flush.zero_()
        layer.forward(x, y)
    st, kms, nc = moe.moe_profile_end(layer.handle)
    assert st == moe.MOE_OK and layer.device_error() == moe.MOE_OK
    layer.close()
    kt = {k: v / nc for k, v in zip(KERNELS_GEMM, kms)}
    ne = int((counts > 0).sum())
    wbytes = (ne * 3 * F * D + 3 * FS * D) * 9 // 16  # 4.5 bits per weight
    layer_bytes = E * D * 2 + wbytes + 2 * T_PREFILL * D * 2
    _, fl, _, layer_flops = algorithmic(counts, T_PREFILL)
    t = ms / 1e3
    t_x = kt["experts"] / 1e3
    return {"ms": ms, "tokens_per_s": T_PREFILL / t, "algorithmic_bytes": layer_bytes,
            "hbm_frac": layer_bytes / t / 1e9 / P_hbm,
            "tensor_frac": layer_flops / t / 1e12 / P_tc,
            "experts_tensor_frac": fl["experts"] / t_x / 1e12 / P_tc,
            "kernel_ms": {k: round(v, 5) for k, v in kt.items()},
            "weights": "4-bit codes, group 64, bf16 scale and bias; router bf16; dequantized "
                       "to bf16 in tensor memory inside the grouped GEMM"}


def run_decode_q4(torch, moe, args, seed, P_hbm):
    """Batch-1 decode with 4-bit group-affine experts (group 64, bf16 scale and bias; the
    router bf16) over 40 layers' weights, one CUDA graph: us/layer and HBM GB/s of the
    bytes this routing needs."""
    dims = synth.Dims(d=D, f=F, fs=FS)
    layers, Ws = [], []
    for l in range(args.decode_layers):
        W = q4_device_weights(torch, seed, l, dims)
        Ws.append(W)
        layers.append(moe.MoeLayer(W, 1))
    x = torch.from_numpy(synth.x_rows(seed, 0, 1, D).view(np.int16)).cuda().view(torch.bfloat16)
    ys = [torch.empty_like(x) for _ in layers]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for L, y in zip(layers, ys):
            L.forward(x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for L, y in zip(layers, ys):
            L.forward(x, y)
    for _ in range(max(3, args.warmup)):
        g.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3 / len(layers)
    L0 = layers[0]
    assert moe.moe_profile_begin(L0.handle, 50) == moe.MOE_OK
    for _ in range(50):
        L0.forward(x, ys[0])
    st, kms, nc = moe.moe_profile_end(L0.handle)
    for L in layers:
        assert L.device_error() == moe.MOE_OK
        L.close()
    gbs = DECODE_Q4_BYTES_PER_LAYER / (us * 1e-6) / 1e9
    return {"us_per_layer": us, "GB_per_s": gbs, "bytes_per_layer": DECODE_Q4_BYTES_PER_LAYER,
            "hbm_frac": gbs / P_hbm, "layers": len(layers),
            "kernel_us_eager": decode_kernel_times(kms, nc),
            "weights": "4-bit codes, group 64, bf16 scale and bias; router bf16"}


def read_probe(torch, moe):
    """GB/s of a read-only stream over 4 GiB (moe_read_probe; a pure read can run faster than
    the copy the measured peak comes from): the best of 10, CUDA events."""
    nbytes = 4 << 30
    buf = torch.ones(nbytes // 2, dtype=torch.bfloat16, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert moe.moe_read_probe(buf.data_ptr(), nbytes, sink.data_ptr(), s) == moe.MOE_OK
    best = None
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        moe.moe_read_probe(buf.data_ptr(), nbytes, sink.data_ptr(), s)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del buf
    return nbytes / (best / 1e3) / 1e9


SMALL_BATCH_T = (2, 3, 4, 5)


def run_small_batch(torch, moe, args, Ws, seed, P_hbm):
    """Decode of T = 2..5 tokens per layer (the speculative-verify shape) over the same 40
    layers' weights, one CUDA graph per T and schedule: us/layer through the matrix-vector
    path over the union of the tokens' experts (schedule GEMV), through the tensor-core path
    (schedule GEMM) and through the default (AUTO: one single-token pass per token at T = 2,
    the tensor-core path above), and the HBM fraction of the bytes this routing needs
    (gate/up/down of the union of the tokens' experts, router, shared expert, x and y) for the
    fastest."""
    out = []
    for T in SMALL_BATCH_T:
        x = torch.from_numpy(synth.x_rows(seed, 0, T, D).view(np.int16)).cuda() \
            .view(torch.bfloat16)
        row = {"T": T}
        for name, sched in (("gemv", moe.MOE_SCHEDULE_GEMV), ("tensor_core", moe.MOE_SCHEDULE_GEMM),
                            ("auto", moe.MOE_SCHEDULE_AUTO)):
            layers = [moe.MoeLayer(W, T, schedule=sched) for W in Ws]
            ys = [torch.empty_like(x) for _ in layers]
            if name == "gemv":
                union = [len(np.unique(L.route(x)["topk_idx"].cpu().numpy())) for L in layers]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for L, y in zip(layers, ys):
                    L.forward(x, y)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for L, y in zip(layers, ys):
                    L.forward(x, y)
            for _ in range(3):
                g.replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(min(args.steps, 50))]
            torch.cuda.synchronize()
            for a, b in ev:
                a.record()
                g.replay()
                b.record()
            torch.cuda.synchronize()
            row[f"{name}_us_per_layer"] = \
                statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3 / len(layers)
            for L in layers:
                assert L.device_error() == moe.MOE_OK
                L.close()
            del g
        nbytes = (statistics.mean(union) * 3 * F * D * 2 + 3 * FS * D * 2 + E * D * 2
                  + 2 * T * D * 2)
        best = min(row["gemv_us_per_layer"], row["tensor_core_us_per_layer"],
                   row["auto_us_per_layer"])
        row.update({"union_experts": statistics.mean(union), "bytes_per_layer": nbytes,
                    "hbm_frac": nbytes / (best * 1e-6) / 1e9 / P_hbm})
        out.append(row)
    return out


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on the
    current source of that kernel (profiles/traffic.txt lines: kernel bytes source-sha)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"router_topk": "route.cu", "route_plan_scatter": "route.cu",
           "experts": "experts.cu", "combine": "experts.cu", "gdn_scan": "gdn.cu"}.get(kernel)
    if not src:
        return None
    sha = hashlib.sha1(open(os.path.join(ROOT, "sparse_moe_02_gb300", "csrc", src), "rb")
                       .read()).hexdigest()[:12]
    for ln in open(path):
        f = ln.split()
        if len(f) >= 3 and f[0] == kernel and f[2] == sha:
            return float(f[1])
    return None


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(torch, world, v, device="cuda"):
    """The largest v over the ranks (the step time of the slowest rank)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, tokens_per_rank, ms):
    """Whole-job tokens/s: every rank runs its own batch of tokens_per_rank tokens (weak
    scaling); ms is the slowest rank's step time."""
    return world * tokens_per_rank / (ms / 1e3)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    import torch
    import sparse_moe_02_gb300 as moe
    moe.lib()  # fail loudly if the CUDA library is not built
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    P_hbm, P_tc, note = peaks()
    clocks = ClockSampler(gpu_smi_id(torch, local))
    clocks.start()
    if args.no_prefill:
        dec = run_decode(torch, moe, args, rank, world, P_hbm)
        clk = clocks.stop()
        if rank == 0:
            print(json.dumps({"decode": dec, "clocks": clk}), flush=True)
        return
    pre = run_prefill(torch, moe, args, rank, world, P_hbm, P_tc, note)
    skewed = None if args.no_skew else time_prefill(
        torch, moe, T_PREFILL, True, min(args.steps, 50), max(3, args.warmup), rank, P_hbm, P_tc)
    sweep = None
    if not args.no_sweep:
        ts = [int(t) for t in args.sweep_tokens.split(",")] if args.sweep_tokens else SWEEP_T
        sweep = [time_prefill(torch, moe, t, False, min(args.steps, 20), 3, rank, P_hbm, P_tc)
                 for t in ts]
        if args.sweep_q4:
            sweep += [time_prefill(torch, moe, t, False, min(args.steps, 20), 3, rank, P_hbm,
                                   P_tc, q4=True) for t in ts]
    pre_q4 = None if args.no_q4 else run_prefill_q4(torch, moe, args, rank, P_hbm, P_tc)
    dec = None if args.no_decode else run_decode(torch, moe, args, rank, world, P_hbm)
    gdn = None if args.no_gdn else run_gdn(torch, moe, args, P_hbm, rank, world)
    clk = clocks.stop()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, sample, cores = oracle_sample_rate(args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": sample}
    if rank != 0:
        return
    value = job_value(world, T_PREFILL, pre["ms"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": pre["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "prefill T=4096 d=2048 E=256 top-8 f=512 + shared (balanced)",
                   "T": T_PREFILL, "d": D, "experts": E, "top_k": K, "ffn_dim": F,
                   "shared_ffn_dim": FS, "parallelism": f"dp{world} (independent batches)",
                   "l2": "flushed (256 MB write, untimed) before every timed step; weights "
                         "1.62 GB > L2"},
        "roofline": pre["roofline"],
        "layer": pre["layer"],
        "prefill_skewed": skewed,
        "prefill_sweep": sweep,
        "prefill_q4": pre_q4,
        "decode": dec,
        "gdn_scan": gdn,
        "cpu_baseline": cpu,
        "e2e": {"value": job_value(world, T_PREFILL, pre["e2e_ms"]), "unit": "tokens/s",
                "h2d_bytes_per_step": T_PREFILL * D * 2, "d2h_bytes_per_step": T_PREFILL * D * 2},
        "gpu_launches": args.steps * pre["launches"],
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
