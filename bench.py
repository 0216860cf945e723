"""Benchmark of the GQA attention hot path on GB300.

Default line: cached single-token decode, Q [1, 32*128], K/V cache
[16384, 8*128] fp32 at kv_pos = 16383 (the whole cache), 32 heads over 8 kv
heads.  Metric: K/V-stream bandwidth in GB/s = algorithmic bytes per step
(K and V window read once, Q read, out written) / device time per step.
Three K/V caches are rotated so each step streams a cache that is not in L2
(3 x 128 MiB > 2 x L2).

The same JSON line carries the prefill (512 queries from start_pos 1536 into
a 2048-row cache, 32 heads over 8, D=128) and long causal forward (q_seq 8192,
32 heads over 8, D=128) results in TFLOP/s, each with its own roofline, and
the CPU oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only other implementation of
the method here) on the host cores for the same metric, on a bounded sample.
Under torchrun each rank runs its own independent decode problem on its own
GPU (no exchange); value = all ranks' bytes / slowest rank's time.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

H, G, D, MAX_SEQ = 32, 8, 128, 16384
KV_POS = 16383
DECODE_WORKLOAD = "decode q[1,32x128] kv_cache[16384,8x128] fp32 kv_pos=16383"
PREFILL = dict(n_queries=512, start_pos=1536, max_seq=2048, H=32, G=8, D=128, stride=4096)
FORWARD = dict(q_seq=8192, H=32, G=8, D=128)
MHA = dict(H=16, D=64, q_full=2048, q_cross=1024, kv_cross=4096)
SWEEP = (0, 7, 511, 4095, 16383)
WINDOW = 4096  # sliding-window workloads: each row keeps its last 4096 keys


def decode_bytes(kv_len):
    return 2 * kv_len * G * D * 4 + 2 * H * D * 4


def prefill_flops():
    p = PREFILL
    tri = sum(p["start_pos"] + i + 1 for i in range(p["n_queries"]))
    return 4.0 * p["D"] * tri * p["H"]


def forward_flops(window=0, q_seq=None):
    """Algorithmic FLOPs of the causal forward: 4 D per (row, head, kept key)."""
    f = FORWARD
    n = q_seq or f["q_seq"]
    keys = n * (n + 1) // 2
    if window:
        w = min(window, n)
        keys = w * (w + 1) // 2 + (n - w) * w
    return 4.0 * f["D"] * keys * f["H"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


def fp32_alu_peak_tflops(sm_mhz, sms):
    # 128 fp32 FMA lanes per SM, 2 flops per FMA.
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def profile_traffic(kernel_tag, src_file):
    """DRAM bytes per launch from the committed ncu summary of `kernel_tag`,
    or None when there is none or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", kernel_tag + ".md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, src_file), "rb").read()).hexdigest()
    return float(m.group(1)) if cur.startswith(h.group(1)) else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, dev_uuid=None):
        self.rows, self.proc, self.th = [], None, None
        self.uuid = dev_uuid

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        rows = [p for (t, p) in self.rows if (t0 is None or t >= t0) and (t1 is None or t <= t1)] or \
            [p for (_, p) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest x over all ranks (x is a host float; the time of the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_step, world, steps, ms_total_max):
    """Whole-job bandwidth in GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_step * world * steps / (ms_total_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------- oracle timing
_ORACLE_INPUTS = {}


def time_oracle_decode(min_seconds, kv_pos=KV_POS):
    """Oracle decode at the bench configuration (window 0..kv_pos), repeated
    for ~min_seconds (at least one call).  Returns (calls, seconds)."""
    import oracle
    from attention_gqa_online_gb300 import synthetic
    orc = oracle.default()
    if not _ORACLE_INPUTS:
        q, kc, vc = synthetic.decode_inputs(MAX_SEQ, H, G, D, seed=0)
        _ORACLE_INPUTS["x"] = (q.numpy(), kc.numpy(), vc.numpy())
    qn, kn, vn = _ORACLE_INPUTS["x"]
    calls, t0 = 0, time.perf_counter()
    while True:
        orc.decode(qn, kn, vn, kv_pos, H, G, D, MAX_SEQ)
        calls += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return calls, el


def decode_config(world):
    """The headline workload, the same for both arms."""
    return {"workload": DECODE_WORKLOAD, "heads": H, "kv_heads": G, "head_dim": D,
            "l2": "inputs larger than 2x L2 between steps (rotating caches)",
            "parallelism": "independent decode per GPU" if world > 1 else "single GPU"}


def reference_arm(args, world, rank):
    """The fp64 CPU oracle on the host cores, same metric and workload.  Each
    step is a bounded sample: the decode over the first n' cache positions,
    n' chosen so the whole run takes about args.ref_seconds."""
    if rank != 0:
        return
    _, t_cal = time_oracle_decode(0.0, kv_pos=1023)          # calibration: 1024 keys
    per_key = t_cal / 1024.0
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n_sample = int(max(64, min(KV_POS + 1, budget / per_key)))
    times = []
    for i in range(args.warmup + args.steps):
        _, el = time_oracle_decode(0.0, kv_pos=n_sample - 1)
        if i >= args.warmup:
            times.append(el)
    per_step = sum(times) / len(times)
    val = decode_bytes(n_sample) / per_step / 1e9
    sample = "per step: oracle decode over cache positions 0..%d (%d of 16384 keys, all 32 heads)" % (
        n_sample - 1, n_sample)
    line = {
        "impl": "reference", "metric": "decode K/V-stream bandwidth", "value": val, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(world),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU arm
def run_ours(args, world, rank, local):
    import torch
    import attention_gqa_online_gb300 as A
    from attention_gqa_online_gb300 import synthetic

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    lib = A.load_library()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    sms = props.multi_processor_count
    peaks, peak_src = load_peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid if rank == 0 else None)
    if rank == 0:
        sampler.start()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # ------------------------------------------------------------------ decode
    cache_bytes = MAX_SEQ * G * D * 4
    n_rot = max(3, int(math.ceil(2.0 * l2 / (2 * cache_bytes))) + 1)
    q, kc, vc = synthetic.decode_inputs(MAX_SEQ, H, G, D, seed=rank)
    qd = q.to(dev)
    caches = [(kc.to(dev), vc.to(dev))]
    for _ in range(n_rot - 1):
        caches.append((caches[0][0].clone(), caches[0][1].clone()))
    out = torch.empty_like(qd)
    ws_bytes = A.attn_decode_workspace_bytes(H, G, D, MAX_SEQ)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    pos = torch.full((1,), KV_POS, dtype=torch.int32, device=dev)
    ptrs = [(k.data_ptr(), v.data_ptr()) for k, v in caches]

    def decode_step(i):
        kp, vp = ptrs[i % n_rot]
        rc = lib.attn_decode_cached(qd.data_ptr(), kp, vp, pos.data_ptr(), out.data_ptr(), H, G, D, MAX_SEQ,
                                    ws.data_ptr(), ws_bytes, sh)
        if rc != 0:
            raise RuntimeError("attn_decode_cached failed: %d" % rc)

    for i in range(args.warmup):
        decode_step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # The timed region is K back-to-back decode launches between two events:
    # the step is one kernel, so its average launch duration in this steady
    # stream (launch and set-up of each step overlap the previous step's tail
    # through programmatic dependent launch) is the timed time / K.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        decode_step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    ms_total = t_start.elapsed_time(t_end)
    kern_ms = ms_total / args.steps
    ms_total = max_over_ranks(ms_total, world)
    # One launch at a time (an event pair around each, nothing to overlap): the
    # kernel's isolated duration, reported beside the steady-state figure.
    iso = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for i in range(50):
        iso[i][0].record(stream)
        decode_step(i)
        iso[i][1].record(stream)
    torch.cuda.synchronize()
    iso_ms = statistics.mean(x.elapsed_time(y) for x, y in iso)
    status = A.attn_get_status(sh)
    if status != 0:
        raise RuntimeError("device status %d after the decode loop" % status)
    ms_step = ms_total / args.steps
    step_bytes = decode_bytes(KV_POS + 1)
    value = weak_scaling_value(step_bytes, world, args.steps, ms_total)
    achieved = step_bytes / (kern_ms * 1e-3) / 1e9
    clocks = sampler.summary(wall0, wall1) if rank == 0 else None

    # e2e: a serving decode step through the public API, its inputs in pinned
    # host memory and its output going back there: attn_decode_append reads
    # [q | k_new | v_new | kv_pos] straight from the pinned buffer (the host
    # link carries them inside the kernel: zero-copy over NVLink-C2C), writes
    # the new K/V row at kv_pos, attends 0..kv_pos, and writes out into pinned
    # host memory.  Eight staging and output buffers rotate, and every step
    # streams the whole K/V window through L2 in between, so each step's bytes
    # cross the link again.
    n_q, n_kv = H * D, G * D
    n_stage = n_q + 2 * n_kv + 4  # kv_pos in the first of four trailing words (16-byte multiple)
    n_io = 8
    stages, outs = [], []
    for b in range(n_io):
        st_h = torch.zeros(n_stage, dtype=torch.float32).pin_memory()
        st_h[:n_q] = q.reshape(-1).cpu()
        st_h[n_q:n_q + n_kv] = caches[0][0][KV_POS].cpu()
        st_h[n_q + n_kv:n_q + 2 * n_kv] = caches[0][1][KV_POS].cpu()
        st_h.view(torch.int32)[n_q + 2 * n_kv] = KV_POS
        stages.append(st_h)
        outs.append(torch.zeros(H * D, dtype=torch.float32).pin_memory())
    h2d = n_stage * 4
    d2h = outs[0].numel() * 4

    def e2e_step(i):
        kd, vd = caches[i % n_rot]
        hp, op = stages[i % n_io].data_ptr(), outs[i % n_io].data_ptr()
        rc = lib.attn_decode_append(hp, hp + 4 * n_q, hp + 4 * (n_q + n_kv), kd.data_ptr(), vd.data_ptr(),
                                    hp + 4 * (n_q + 2 * n_kv), op, H, G, D, MAX_SEQ, ws.data_ptr(), ws_bytes, sh)
        if rc != 0:
            raise RuntimeError("attn_decode_append failed: %d" % rc)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if A.attn_get_status(sh) != 0 or not all(bool(torch.isfinite(o).all()) for o in outs):
        raise RuntimeError("the end-to-end decode steps failed")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_val = step_bytes * world * args.steps / (e2e_ms * 1e-3) / 1e9
    del caches

    extras = {}
    if rank == 0 and not args.decode_only:
        extras = run_extras(args, A, lib, synthetic, dev, stream, sh, l2, sms, peaks, peak_src, clocks)

    if rank == 0:
        sampler.stop()
        traffic = profile_traffic("decode_split_kernel_kvpos16383", "attention_gqa_online_gb300/csrc/decode.cu")
        line = {
            "metric": "decode K/V-stream bandwidth", "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": decode_config(world),
            "l2": "inputs rotate over %d K/V caches (%d MiB) > 2x L2" % (n_rot, n_rot * 2 * cache_bytes >> 20),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "decode_split_kernel<128,4>", "kernel_us": kern_ms * 1e3,
                         "isolated_launch_us": iso_ms * 1e3,
                         "bytes_per_launch": step_bytes, "peak_source": peak_src},
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "what": "per step: attn_decode_append reads [q | new K row | new V row | kv_pos] from pinned "
                            "host memory and writes out to pinned host memory (zero-copy over the host link, 8 "
                            "rotating buffers); it writes the row at kv_pos and attends 0..kv_pos",
                    "us_per_step": e2e_ms * 1e3 / args.steps},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "decode_us_per_token": ms_step * 1e3,
        }
        if not args.no_cpu_baseline:
            calls, el = time_oracle_decode(args.cpu_seconds)
            line["cpu_baseline"] = {"value": decode_bytes(KV_POS + 1) * calls / el / 1e9, "unit": "GB/s",
                                    "cores": 1, "kind": "oracle",
                                    "sample": "%d oracle decode calls at kv_pos=16383 in %.1f s" % (calls, el)}
        line.update(extras)
        line["summary"] = summary(line, extras)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# Order of the compact summary that closes the JSON line (last = most
# important: a reader that keeps only the line's tail still sees them).
SUMMARY_ORDER = ("backward_fp32", "backward_bf16", "forward_rope_fp32", "forward_rope_tf32", "forward_rope_bf16",
                 "forward_window_fp32", "forward_window_tf32", "forward_window_bf16", "decode_window", "decode_gqa8",
                 "decode_paged", "prefill_paged_tf32", "prefill_paged_bf16", "mha_cross_fp32", "mha_cross_tf32",
                 "mha_cross_bf16", "mha_full_fp32", "mha_full_tf32", "mha_full_bf16", "forward_8193_fp32",
                 "forward_8193_tf32", "forward_8193_bf16", "forward_fp32", "forward_tf32", "forward_bf16",
                 "prefill_fp32", "prefill_tf32", "prefill_bf16")


def summary(line, extras):
    """Compact {workload: [value, unit, roofline fraction]} of every line, the
    decode sweep as {kv_pos: [us/token, GB/s]}, and the headline decode last."""
    out = {}
    for k in SUMMARY_ORDER:
        e = extras.get(k)
        if e:
            out[k] = [round(e["value"], 1), e["unit"], round(e["roofline"]["frac"], 3)]
    sw = extras.get("decode_sweep")
    if sw:
        out["decode_sweep_us_GBs"] = {p: [round(x["us_per_token"], 2), round(x["GB/s"], 0)]
                                      for p, x in sw["points"].items()}
    out["decode"] = [round(line["value"], 1), line["unit"], round(line["roofline"]["frac"], 3)]
    return out


def tf32_peak(peaks):
    """TF32 dense peak: the measured bf16 peak times the nominal TF32 / bf16 ratio (1.1 / 2.25)."""
    return peaks["bf16_tflops"] * 1.1 / 2.25


def run_extras(args, A, lib, synthetic, dev, stream, sh, l2, sms, peaks, peak_src, clocks, only="all"):
    """Prefill and long causal forward in TFLOP/s on the TF32 and bf16
    tensor-core paths and the fp32 CUDA-core path."""
    import torch
    res = {"_launches": 0}
    sm_mhz = (clocks or {}).get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    alu_peak = fp32_alu_peak_tflops(sm_mhz, sms)
    steps = max(3, min(args.steps, args.extra_steps))

    def timed(fn, n):
        """Mean device time per call of n back-to-back calls between one event
        pair (each call's kernels chain to the previous call's by programmatic
        dependent launch, as in a stream of calls; an event between calls would
        break that chain).  Inputs rotate over sets larger than L2 together."""
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res["_launches"] += n + args.warmup
        return e0.elapsed_time(e1) / n

    # Committed ncu summaries per (precision, workload): profiles/<tag>.md and
    # the kernel source it was captured from.
    flash_src = {A.ATTN_BF16: ("flash_bf16_kernel", "attention_gqa_online_gb300/csrc/flash_bf16.cu"),
                 A.ATTN_TF32: ("flash_tc_kernel", "attention_gqa_online_gb300/csrc/flash_tc.cu"),
                 A.ATTN_FP32: ("flash_simt_kernel", "attention_gqa_online_gb300/csrc/flash_simt.cu")}

    def roof(prec, tf, kernel, workload=None, prof=None):
        """Roofline of the line's dominant kernel; `traffic` from profiles/<kernel>_<workload>.md
        (or the (tag, source) pair `prof`) when that summary exists and matches the kernel's
        current source."""
        traffic = None
        if prof is not None:
            traffic = profile_traffic(*prof)
        elif workload is not None and prec in flash_src:
            tag, src = flash_src[prec]
            traffic = profile_traffic(tag + "_" + workload, src)
        if prec == A.ATTN_BF16:
            pk = peaks["bf16_tflops"]
            return {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                    "traffic": traffic, "kernel": kernel, "peak_source": "%s bf16 dense, burst" % peak_src}
        if prec == A.ATTN_TF32:
            pk = tf32_peak(peaks)
            return {"bound": "tensor", "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk,
                    "traffic": traffic, "kernel": kernel,
                    "peak_source": "%s bf16 %.0f TFLOP/s x 1.1/2.25 (nominal TF32/bf16)" % (peak_src, peaks["bf16_tflops"])}
        return {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                "traffic": traffic, "kernel": kernel,
                "peak_source": "fp32 FMA: %d SMs x 128 lanes x 2 x %.0f MHz" % (sms, sm_mhz)}

    def forward_lines(prefix, window, what, rope=False, q_seq=None):
        f = dict(FORWARD)
        if q_seq is not None:
            f["q_seq"] = q_seq
        q, k, v = synthetic.forward_inputs(f["q_seq"], f["q_seq"], f["H"], f["G"], f["D"], seed=5, qk_sigma=3.0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        outf = torch.empty_like(qd)
        lse = torch.empty((f["q_seq"], f["H"], 2), device=dev)
        tab = torch.empty((f["q_seq"], f["D"]), device=dev)
        if rope:
            A.attn_rope_table(tab, f["q_seq"], f["D"], 10000.0, stream)
        for prec, name, kern in variants:
            def fwd_step(i, prec=prec):
                if rope:
                    rc = lib.attn_forward_rope(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outf.data_ptr(),
                                               lse.data_ptr(), f["q_seq"], f["q_seq"], f["H"], f["G"], f["D"],
                                               A.ATTN_CAUSAL, prec, window, tab.data_ptr(), f["q_seq"], sh)
                else:
                    rc = lib.attn_forward_window(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outf.data_ptr(),
                                                 lse.data_ptr(), f["q_seq"], f["q_seq"], f["H"], f["G"], f["D"],
                                                 A.ATTN_CAUSAL, prec, window, sh)
                if rc != 0:
                    raise RuntimeError("forward failed: %d" % rc)
            ms = timed(fwd_step, steps)
            tf = forward_flops(window, f["q_seq"]) / (ms * 1e-3) / 1e12
            plain = not rope and not window and q_seq is None
            res[prefix + name] = {
                "workload": what, "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "prec": name,
                "roofline": roof(prec, tf, kern, "forward_q8192" if plain else None), "l2": "inputs 192 MiB > L2"}

    variants = ((A.ATTN_TF32, "tf32", "flash_tc_kernel<128> (tf32)"),
                (A.ATTN_BF16, "bf16", "flash_bf16_kernel<128> (fp16 QK, bf16 PV) + kv_prep16 pre-pass"),
                (A.ATTN_FP32, "fp32", "flash_simt_kernel<128,true>"))

    if only in ("all", "prefill"):
        p = PREFILL
        qb, kc, vc = synthetic.prefill_inputs(p["n_queries"], p["stride"], p["max_seq"], p["G"] * p["D"], seed=0)
        per = (qb.numel() + kc.numel() + vc.numel()) * 4
        n_rot = max(2, int(math.ceil(2.0 * l2 / per)) + 1)
        bufs = [(qb.to(dev), kc.to(dev), vc.to(dev)) for _ in range(n_rot)]
        outp = torch.empty((p["n_queries"], p["stride"]), device=dev)
        scale = 1.0 / math.sqrt(p["D"])
        for prec, name, kern in variants:
            def prefill_step(i, prec=prec):
                qd, kd, vd = bufs[i % n_rot]
                rc = lib.attn_prefill(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outp.data_ptr(), p["n_queries"],
                                      p["H"], p["G"], p["D"], p["G"] * p["D"], p["max_seq"], scale, p["start_pos"],
                                      p["stride"], p["stride"], 0, prec, sh)
                if rc != 0:
                    raise RuntimeError("attn_prefill failed: %d" % rc)
            ms = timed(prefill_step, steps)
            tf = prefill_flops() / (ms * 1e-3) / 1e12
            res["prefill_" + name] = {
                "workload": "prefill 512 queries start_pos=1536 max_seq=2048 32/8 heads D=128",
                "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "prec": name,
                "roofline": roof(prec, tf, kern, "prefill_512q"), "l2": "rotating %d input sets" % n_rot}
        del bufs

    if only in ("all", "forward"):
        forward_lines("forward_", 0, "causal forward+LSE q_seq=8192 32/8 heads D=128, Q,K N(0,9)")

    if only in ("all", "rope"):
        forward_lines("forward_rope_", 0, "causal forward+LSE with RoPE on q and k (base 10000), q_seq=8192 32/8 "
                      "heads D=128, Q,K N(0,9)", rope=True)

    if only in ("all", "backward"):
        # fp32 backward of the long causal forward (dq, dk, dv from out, lse, dout).
        f = FORWARD
        q, k, v = synthetic.forward_inputs(f["q_seq"], f["q_seq"], f["H"], f["G"], f["D"], seed=5, qk_sigma=3.0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        outf = torch.empty_like(qd)
        lse = torch.empty((f["q_seq"], f["H"], 2), device=dev)
        rc = lib.attn_forward(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outf.data_ptr(), lse.data_ptr(),
                              f["q_seq"], f["q_seq"], f["H"], f["G"], f["D"], A.ATTN_CAUSAL, A.ATTN_FP32, sh)
        if rc != 0:
            raise RuntimeError("attn_forward failed: %d" % rc)
        gout = torch.randn(qd.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(3))
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        bwd_prof = {A.ATTN_BF16: ("bwd_dkdv_tc_kernel_backward_q8192", "attention_gqa_online_gb300/csrc/bwd_tc.cu"),
                    A.ATTN_FP32: ("bwd_dkdv_kernel_backward_q8192", "attention_gqa_online_gb300/csrc/backward.cu")}
        for prec, name, kern, nsteps in (
                (A.ATTN_BF16, "bf16", "bwd_dkdv_tc_kernel<128> + bwd_dq_tc_kernel<128> (+ prep, bf16 pre-passes)",
                 steps),
                (A.ATTN_FP32, "fp32", "bwd_dkdv_kernel<128> + bwd_dq_kernel<128> (+ bwd_prep_kernel)",
                 max(3, steps // 4))):
            def bwd_step(i, prec=prec):
                rc = lib.attn_backward(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outf.data_ptr(), gout.data_ptr(),
                                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), f["q_seq"],
                                       f["q_seq"], f["H"], f["G"], f["D"], A.ATTN_CAUSAL, prec, 0, sh)
                if rc != 0:
                    raise RuntimeError("attn_backward failed: %d" % rc)
            ms = timed(bwd_step, nsteps)
            tf = 2.5 * forward_flops() / (ms * 1e-3) / 1e12
            res["backward_" + name] = {
                "workload": "causal backward (dq, dk, dv) q_seq=8192 32/8 heads D=128, Q,K N(0,9)", "value": tf,
                "unit": "TFLOP/s", "ms_per_step": ms, "prec": name,
                "flops": "2.5x the forward's: 10 D per (row, head, kept key), the five products of the gradient",
                "roofline": roof(prec, tf, kern, prof=bwd_prof[prec]), "l2": "inputs 320 MiB > L2"}
        del qd, kd, vd, outf, gout, dq, dk, dv

    if only in ("all", "paged"):
        # Paged cache: the decode and prefill workloads with their caches cut
        # into pages placed in shuffled order in a pool.
        P_DEC, P_PRE = 64, 128
        nb = MAX_SEQ // P_DEC
        rng = torch.Generator().manual_seed(11)
        q, kc, vc = synthetic.decode_inputs(MAX_SEQ, H, G, D, seed=1)
        qd = q.to(dev)
        cache_bytes = 2 * MAX_SEQ * G * D * 4
        n_rot = max(3, int(math.ceil(2.0 * l2 / cache_bytes)) + 1)
        pools, tables = [], []
        for r in range(n_rot):
            perm = torch.randperm(nb, generator=rng)
            pools.append((kc.view(nb, P_DEC, G * D)[perm].reshape(MAX_SEQ, G * D).to(dev),
                          vc.view(nb, P_DEC, G * D)[perm].reshape(MAX_SEQ, G * D).to(dev)))
            tables.append(torch.argsort(perm).to(torch.int32).to(dev))  # logical page b -> pool page
        out = torch.empty_like(qd)
        ws_bytes = A.attn_decode_workspace_bytes(H, G, D, MAX_SEQ)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        pos = torch.full((1,), KV_POS, dtype=torch.int32, device=dev)

        def pdec_step(i):
            kd, vd = pools[i % n_rot]
            rc = lib.attn_decode_paged(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), tables[i % n_rot].data_ptr(),
                                       pos.data_ptr(), out.data_ptr(), H, G, D, P_DEC, nb, nb, ws.data_ptr(),
                                       ws_bytes, 0, sh)
            if rc != 0:
                raise RuntimeError("attn_decode_paged failed: %d" % rc)
        for i in range(args.warmup):
            pdec_step(i)
        torch.cuda.synchronize()
        n_dec = max(steps, 200)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_dec):
            pdec_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res["_launches"] += n_dec + args.warmup
        ms = e0.elapsed_time(e1) / n_dec
        by = decode_bytes(KV_POS + 1)
        gbs = by / (ms * 1e-3) / 1e9
        res["decode_paged"] = {
            "workload": "decode kv_pos=16383, cache of 256 pages x 64 rows in shuffled pool order, [16384, 8x128] fp32",
            "value": gbs, "unit": "GB/s", "us_per_step": ms * 1e3,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "decode_split_kernel<128,4>",
                         "bytes_per_launch": by, "peak_source": peak_src},
            "l2": "rotating %d pools > 2x L2" % n_rot, "timing": "%d back-to-back launches" % n_dec}
        del pools
        pp = PREFILL
        nbp = pp["max_seq"] // P_PRE
        qb, kc2, vc2 = synthetic.prefill_inputs(pp["n_queries"], pp["stride"], pp["max_seq"], pp["G"] * pp["D"], seed=0)
        per = (qb.numel() + kc2.numel() + vc2.numel()) * 4
        n_rot2 = max(2, int(math.ceil(2.0 * l2 / per)) + 1)
        bufs = []
        for r in range(n_rot2):
            perm = torch.randperm(nbp, generator=rng)
            bufs.append((qb.to(dev), kc2.view(nbp, P_PRE, -1)[perm].reshape(pp["max_seq"], -1).to(dev),
                         vc2.view(nbp, P_PRE, -1)[perm].reshape(pp["max_seq"], -1).to(dev),
                         torch.argsort(perm).to(torch.int32).to(dev)))
        outp = torch.empty((pp["n_queries"], pp["stride"]), device=dev)
        scale = 1.0 / math.sqrt(pp["D"])
        for prec, name, kern in variants[:2]:
            def pprefill_step(i, prec=prec):
                qd2, kd, vd, td = bufs[i % n_rot2]
                rc = lib.attn_prefill_paged(qd2.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(), outp.data_ptr(),
                                            pp["n_queries"], pp["H"], pp["G"], pp["D"], pp["G"] * pp["D"], P_PRE, nbp,
                                            nbp, scale, pp["start_pos"], pp["stride"], pp["stride"], 0, prec, 0, sh)
                if rc != 0:
                    raise RuntimeError("attn_prefill_paged failed: %d" % rc)
            ms = timed(pprefill_step, steps)
            tf = prefill_flops() / (ms * 1e-3) / 1e12
            res["prefill_paged_" + name] = {
                "workload": "prefill 512 queries start_pos=1536, cache of 16 pages x 128 rows in shuffled pool order, "
                            "32/8 heads D=128", "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "prec": name,
                "roofline": roof(prec, tf, kern + (" (gathering the pages)" if prec == A.ATTN_BF16 else "")),
                "l2": "rotating %d input sets" % n_rot2}
        del bufs

    if only in ("all", "decode_gqa8"):
        # 64 query heads over 8 kv heads at D = 128 (two head groups per kv head).
        H8 = 64
        q8, kc8, vc8 = synthetic.decode_inputs(MAX_SEQ, H8, G, D, seed=2)
        q8d = q8.to(dev)
        n_rot8 = max(3, int(math.ceil(2.0 * l2 / (2 * MAX_SEQ * G * D * 4))) + 1)
        caches8 = [(kc8.to(dev), vc8.to(dev)) for _ in range(n_rot8)]
        out8 = torch.empty_like(q8d)
        ws8_bytes = A.attn_decode_workspace_bytes(H8, G, D, MAX_SEQ)
        ws8 = torch.zeros(ws8_bytes, dtype=torch.uint8, device=dev)
        pos8 = torch.full((1,), KV_POS, dtype=torch.int32, device=dev)

        def dec8_step(i):
            kd, vd = caches8[i % n_rot8]
            rc = lib.attn_decode_cached(q8d.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos8.data_ptr(), out8.data_ptr(),
                                        H8, G, D, MAX_SEQ, ws8.data_ptr(), ws8_bytes, sh)
            if rc != 0:
                raise RuntimeError("attn_decode_cached failed: %d" % rc)
        for i in range(args.warmup):
            dec8_step(i)
        torch.cuda.synchronize()
        n_dec = max(steps, 200)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_dec):
            dec8_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res["_launches"] += n_dec + args.warmup
        ms = e0.elapsed_time(e1) / n_dec
        by = 2 * (KV_POS + 1) * G * D * 4 + 2 * H8 * D * 4
        gbs = by / (ms * 1e-3) / 1e9
        res["decode_gqa8"] = {
            "workload": "decode q[1,64x128] kv_cache[16384,8x128] fp32 kv_pos=16383 (8 query heads per kv head)",
            "value": gbs, "unit": "GB/s", "us_per_step": ms * 1e3,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                         "kernel": "decode_split_kernel<128,4> x 2 head groups per kv head",
                         "bytes_per_launch": by, "peak_source": peak_src},
            "l2": "rotating %d caches > 2x L2" % n_rot8, "timing": "%d back-to-back launches" % n_dec}
        del caches8

    if only in ("all", "window"):
        forward_lines("forward_window_", WINDOW, "sliding-window causal forward+LSE q_seq=8192 window=%d 32/8 heads "
                      "D=128, Q,K N(0,9)" % WINDOW)
        # Windowed decode: the last WINDOW positions of a 16384-row cache.
        win_bytes = decode_bytes(WINDOW)
        n_rot = max(3, int(math.ceil(2.0 * l2 / (win_bytes - 2 * H * D * 4))) + 1)
        q, kc, vc = synthetic.decode_inputs(MAX_SEQ, H, G, D, seed=1)
        qd = q.to(dev)
        caches = [(kc.to(dev), vc.to(dev)) for _ in range(n_rot)]
        out = torch.empty_like(qd)
        ws_bytes = A.attn_decode_workspace_bytes(H, G, D, MAX_SEQ)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        pos = torch.full((1,), KV_POS, dtype=torch.int32, device=dev)

        def dec_step(i):
            kd, vd = caches[i % n_rot]
            rc = lib.attn_decode_cached_window(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos.data_ptr(),
                                               out.data_ptr(), H, G, D, MAX_SEQ, ws.data_ptr(), ws_bytes, WINDOW, sh)
            if rc != 0:
                raise RuntimeError("attn_decode_cached_window failed: %d" % rc)
        # Back-to-back launches between one event pair, as for the main
        # decode line (each launch overlaps the previous one's tail by PDL).
        for i in range(args.warmup):
            dec_step(i)
        torch.cuda.synchronize()
        n_dec = max(steps, 200)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_dec):
            dec_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res["_launches"] += n_dec + args.warmup
        ms = e0.elapsed_time(e1) / n_dec
        gbs = win_bytes / (ms * 1e-3) / 1e9
        res["decode_window"] = {
            "workload": "decode kv_pos=16383 window=%d (positions 12288..16383), cache [16384, 8x128] fp32" % WINDOW,
            "value": gbs, "unit": "GB/s", "us_per_step": ms * 1e3,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "decode_split_kernel<128,4>",
                         "bytes_per_launch": win_bytes, "peak_source": peak_src},
            "l2": "rotating %d caches (%d MiB of windows) > 2x L2" % (n_rot, n_rot * (win_bytes >> 20)),
            "timing": "%d back-to-back launches between one event pair" % n_dec}
        del caches

    if only in ("all", "forward"):
        # The long causal stress workload's ragged length.
        forward_lines("forward_8193_", 0, "causal forward+LSE q_seq=8193 (ragged last tile) 32/8 heads D=128, "
                      "Q,K N(0,9)", q_seq=8193)

    if only in ("all", "mha"):
        # Full and cross attention, 16 heads = 16 kv heads, D=64, Q,K N(0,1), V U(-1,1).
        for name, mask, qs, ks in (("mha_full_", A.ATTN_FULL, MHA["q_full"], MHA["q_full"]),
                                   ("mha_cross_", A.ATTN_CROSS, MHA["q_cross"], MHA["kv_cross"])):
            q, k, v = synthetic.forward_inputs(qs, ks, MHA["H"], MHA["H"], MHA["D"], seed=4, v_dist="uniform")
            per = (q.numel() + k.numel() + v.numel()) * 4 * 2
            n_rot = max(2, int(math.ceil(2.0 * l2 / per)) + 1)
            bufs = [(q.to(dev), k.to(dev), v.to(dev)) for _ in range(n_rot)]
            outm = torch.empty_like(bufs[0][0])
            lsem = torch.empty((qs, MHA["H"], 2), device=dev)
            flops = 4.0 * MHA["D"] * qs * ks * MHA["H"]
            what = "%s forward+LSE q=%d kv=%d, 16/16 heads D=64, Q,K N(0,1), V U(-1,1)" % (
                "full" if mask == A.ATTN_FULL else "cross", qs, ks)
            kern = {A.ATTN_TF32: "flash_tc_kernel<64> (tf32)", A.ATTN_BF16: "flash_bf16_kernel<64> + kv_prep16",
                    A.ATTN_FP32: "flash_simt_kernel<64>"}
            for prec, pname in ((A.ATTN_TF32, "tf32"), (A.ATTN_BF16, "bf16"), (A.ATTN_FP32, "fp32")):
                def mha_step(i, prec=prec, mask=mask, qs=qs, ks=ks):
                    qd, kd, vd = bufs[i % n_rot]
                    rc = lib.attn_forward(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), outm.data_ptr(),
                                          lsem.data_ptr(), qs, ks, MHA["H"], MHA["H"], MHA["D"], mask, prec, sh)
                    if rc != 0:
                        raise RuntimeError("attn_forward failed: %d" % rc)
                ms = timed(mha_step, steps)
                tf = flops / (ms * 1e-3) / 1e12
                res[name + pname] = {"workload": what, "value": tf, "unit": "TFLOP/s", "ms_per_step": ms,
                                     "prec": pname, "roofline": roof(prec, tf, kern[prec]),
                                     "l2": "rotating %d input sets" % n_rot}
            del bufs

    if only in ("all", "sweep"):
        # Decode at every kv_pos of the sweep: microseconds per token and K/V GB/s.
        q, kc, vc = synthetic.decode_inputs(MAX_SEQ, H, G, D, seed=3)
        qd = q.to(dev)
        n_rot = max(3, int(math.ceil(2.0 * l2 / (2 * MAX_SEQ * G * D * 4))) + 1)
        caches = [(kc.to(dev), vc.to(dev)) for _ in range(n_rot)]
        out = torch.empty_like(qd)
        ws_bytes = A.attn_decode_workspace_bytes(H, G, D, MAX_SEQ)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        pos = torch.zeros((1,), dtype=torch.int32, device=dev)
        sweep = {}
        for kv_pos in SWEEP:
            pos.fill_(kv_pos)

            def sw_step(i):
                kd, vd = caches[i % n_rot]
                rc = lib.attn_decode_cached(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos.data_ptr(),
                                            out.data_ptr(), H, G, D, MAX_SEQ, ws.data_ptr(), ws_bytes, sh)
                if rc != 0:
                    raise RuntimeError("attn_decode_cached failed: %d" % rc)
            for i in range(args.warmup):
                sw_step(i)
            torch.cuda.synchronize()
            n_dec = max(steps, 200)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n_dec):
                sw_step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            res["_launches"] += n_dec + args.warmup
            ms = e0.elapsed_time(e1) / n_dec
            by = decode_bytes(kv_pos + 1)
            gbs = by / (ms * 1e-3) / 1e9
            sweep[str(kv_pos)] = {"us_per_token": ms * 1e3, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"],
                                  "bytes": by}
        res["decode_sweep"] = {
            "workload": "decode q[1,32x128] kv_cache[16384,8x128] fp32 at kv_pos in %s" % (list(SWEEP),),
            "points": sweep, "unit": "us/token and GB/s", "kernel": "decode_split_kernel<128,4>",
            "peak": peaks["hbm_gbs"], "peak_source": peak_src, "l2": "rotating %d caches > 2x L2" % n_rot,
            "timing": "%d back-to-back launches per point" % max(steps, 200)}
        del caches
    return res


def run_single(args, local):
    """Prefill or forward workloads only (for profiling)."""
    import torch
    import attention_gqa_online_gb300 as A
    from attention_gqa_online_gb300 import synthetic
    torch.cuda.set_device(local)
    lib = A.load_library()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)
    res = run_extras(args, A, lib, synthetic, dev, stream, stream.cuda_stream,
                     getattr(props, "L2_cache_size", 128 << 20), props.multi_processor_count, peaks, peak_src,
                     None, only=args.only)
    res.pop("_launches", None)
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--decode-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["all", "decode", "prefill", "forward", "window", "backward", "paged", "rope",
                                       "decode_gqa8", "mha", "sweep"],
                    default="all",
                    help="run one workload (for profiling); the default runs all of them")
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    if args.only in ("prefill", "forward", "window", "backward", "paged", "rope", "decode_gqa8", "mha", "sweep"):
        run_single(args, local)
        return
    if args.only == "decode":
        args.decode_only = True
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
