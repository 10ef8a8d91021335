#!/usr/bin/env python3
"""KDA forward benchmark on GB300.

One step = one chunked prefill of the T = 65536, H = 32, d = 128 problem
(B = 1, random fp32 initial state) through the C-ABI library, inputs resident
in HBM.  The same run also measures the decode step (256 sequences x 32
heads, 1000 chained in-place steps) and reports it beside the headline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun (N > 1) every rank runs its
own copy of the problem on its own GPU (independent heads/sequences: no
collective on the data path), timings are maxed over ranks and `value` is
the aggregate.  `--impl reference` times the fp64 CPU oracle on the host's
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill Mtok/s & % BF16 tensor peak at T=64k; decode state GB/s % HBM"
FLOP_PER_TOKEN_HEAD = 2 * (5 * 64 * 128 + 3 * 128 * 128)  # 180224, chunk 64, d 128
L2_BYTES = 126 * 2 ** 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def prefill_bytes(tokens, H, d, out_bytes, n_states):
    """Compulsory HBM bytes of one prefill: q, k, v, log_alpha (bf16), beta
    (bf16), the output, and the fp32 state read and written once.  With a
    bf16 output this is 1282 B per token-head at d = 128 (the roofline's unit
    of work); the fp32 output this benchmark writes adds 256 B."""
    return tokens * H * (4 * d * 2 + 2 + d * out_bytes) + 2 * n_states * H * d * d * 4


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"kda_clocks_{os.getpid()}.csv")
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = ["-i", str(device_index)]

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl)
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def source_code(text):
    """The code of a C/CUDA source: comments, indentation and blank lines
    removed, so that a comment edit leaves the hash below unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_hash():
    """Hash of the prefill kernels' code (not their comments)."""
    h = hashlib.sha256()
    for f in ("kda_chunk.cu", "umma.cuh"):
        path = os.path.join(ROOT, "linear_attention_recurrence_fwd_gb300", "csrc", f)
        h.update(source_code(open(path).read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else null)."""
    p = os.path.join(ROOT, "profiles", "chunk_prefill_traffic.json")
    try:
        d = json.load(open(p))
        if d.get("kernel_sha") == kernel_hash():
            return float(d["dram_bytes_per_launch_full_size"])
    except Exception:
        pass
    return None


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def reduce_max(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample(x, heads, threads=0):
    """Time the fp64 oracle on `heads` heads of the full-length problem."""
    from oracle import oracle as orc

    sub = {k: x[k][:, :, :heads].cpu() for k in ("q", "k", "v", "log_alpha", "beta")}
    s0 = x["initial_state"][:, :heads].cpu() if x["initial_state"] is not None else None
    t0 = time.perf_counter()
    orc.kda_recurrence(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"], s0,
                       threads=threads)
    return time.perf_counter() - t0, orc.max_threads()


REF_HEADS = 4  # heads of the T = 65536 problem the reference arm runs per step


def run_reference(args, ws, rank):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores.
    Each step is a bounded sample of the T = 65536, H = 32 problem: REF_HEADS
    heads over all 65536 tokens.  `ms_per_step` is the time of that sample as
    measured; `value` counts the sample's work in whole-problem tokens
    (65536 * REF_HEADS / 32 per step), so it is the rate the oracle would
    reach on the full problem."""
    if rank != 0:
        return
    from linear_attention_recurrence_fwd_gb300 import inputs as gen

    w = gen.WORKLOADS["prefill_64k"]
    x = gen.make_inputs(1, w.T, REF_HEADS, w.dk, w.dv, w.seed, w.decay_mean, w.init_std)
    for _ in range(args.warmup):
        oracle_sample(x, REF_HEADS)
    times = []
    cores = 1
    for _ in range(args.steps):
        t, cores = oracle_sample(x, REF_HEADS)
        times.append(t)
    sec = statistics.mean(times)
    value = w.T * REF_HEADS / w.H / sec / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mtok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill_64k: B=1 T=65536 H=32 d=128", "B": 1, "T": w.T,
                   "H": w.H, "d": w.dk},
        "cpu_baseline": {"value": value, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": f"{REF_HEADS} of {w.H} heads, all {w.T} tokens, per step "
                                   f"(ms_per_step is the sample's time)"},
        "e2e": {"value": value, "unit": "Mtok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_call(fn, steps, warmup, stream):
    """Average CUDA-event milliseconds of fn() over `steps` calls on `stream`."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def extra_workloads(args, ws, dev, stream, x64, ms64):
    """The other prefill shapes, timed the same way (inputs resident, larger
    than L2), plus the per-pair diagonal ablation on the T = 65536 problem."""
    from linear_attention_recurrence_fwd_gb300 import binding
    from linear_attention_recurrence_fwd_gb300 import inputs as gen

    res = {}
    a64 = [x64[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    out = torch.empty(x64["v"].shape, dtype=torch.float32, device=dev)
    fin = torch.empty_like(x64["initial_state"])

    def ablation():
        binding.kda_chunk_fwd(*a64, x64["initial_state"], out=out, final_state=fin)

    os.environ["KDA_ABLATE_DIAG"] = "1"
    try:
        ms = reduce_max(time_call(ablation, 5, 3, stream), ws)
    finally:
        del os.environ["KDA_ABLATE_DIAG"]
    tok = x64["q"].shape[0] * x64["q"].shape[1]
    res["ablation_diag_per_pair"] = {
        "workload": "prefill_64k with the diagonal tiles evaluated per position pair",
        "ms": ms, "Mtok_s": ws * tok / ms / 1e3, "slowdown_vs_dense": ms / ms64, "steps": 5}
    # the same problem saving the state every 512 tokens (a prefix cache)
    ck = torch.empty((1, x64["q"].shape[1] // 512, x64["q"].shape[2], 128, 128),
                     dtype=torch.float32, device=dev)
    ms_ck = reduce_max(time_call(lambda: binding.kda_chunk_fwd_checkpointed(
        *a64, x64["initial_state"], checkpoint_every=512, out=out, final_state=fin,
        checkpoints=ck), 10, 3, stream), ws)
    res["prefill_64k_checkpoints_512"] = {
        "workload": "prefill_64k, state saved every 512 tokens "
                    f"({ck.shape[1]} x {ck.shape[2]} heads x 64 KiB)",
        "ms": ms_ck, "Mtok_s": ws * tok / ms_ck / 1e3, "overhead_vs_plain": ms_ck / ms64 - 1,
        "steps": 10}
    del out, fin, a64, ck

    def fixed(name, steps):
        w = gen.WORKLOADS[name]
        x = gen.workload_inputs(w, device=dev)
        a = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
        o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.float32, device=dev)
        f = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
        s0 = x["initial_state"] if w.init_std > 0 else None
        ms = reduce_max(time_call(
            lambda: binding.kda_chunk_fwd(*a, s0, out=o, final_state=f), steps, 3, stream), ws)
        res[name] = {"workload": f"B={w.B} T={w.T} H={w.H} d={w.dk}", "ms": ms,
                     "Mtok_s": ws * w.B * w.T / ms / 1e3, "steps": steps}

    fixed("prefill_8k", 20)

    # backward of the 8k prefill (training): the forward again for the state
    # at every chunk boundary, then the reverse token recurrence
    w = gen.WORKLOADS["prefill_8k"]
    x = gen.workload_inputs(w, device=dev)
    a = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    d_out = torch.randn((w.B, w.T, w.H, w.dv), dtype=torch.float32, device=dev,
                        generator=torch.Generator(device=dev).manual_seed(w.seed + 1))
    ms = reduce_max(time_call(lambda: binding.kda_chunk_bwd(
        *a, d_out, initial_state=x["initial_state"]), 5, 2, stream), ws)
    res["backward_8k"] = {"workload": f"gradients of prefill_8k (B={w.B} T={w.T} H={w.H} "
                                      f"d={w.dk}) for a random d_out, fp32",
                          "ms": ms, "Mtok_s": ws * w.B * w.T / ms / 1e3,
                          "forward_ms": res["prefill_8k"]["ms"], "steps": 5}
    del x, a, d_out

    # speculative decoding: verify 4 drafted tokens per sequence (state read
    # once), then commit all 4 (state read and written once)
    wd = gen.WORKLOADS["decode"]
    K = 4
    xd = gen.make_inputs(wd.B, K, wd.H, 128, 128, wd.seed, init_std=wd.init_std, device=dev)
    dd = [xd[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    st = xd["initial_state"]
    vo = torch.empty((wd.B, K, wd.H, 128), dtype=torch.float32, device=dev)
    acc = torch.full((wd.B,), K, dtype=torch.int32, device=dev)
    ms_v = reduce_max(time_call(lambda: binding.kda_decode_verify(*dd, st, out=vo), 50, 3,
                                stream), ws)
    ms_c = reduce_max(time_call(lambda: binding.kda_decode_commit(*dd, st, acc), 50, 3, stream),
                      ws)
    sbytes = wd.B * wd.H * 128 * 128 * 4
    io = wd.B * K * wd.H * (4 * 128 * 2 + 2)
    res["speculative_verify_commit_k4"] = {
        "workload": f"{wd.B} seq x {wd.H} heads, {K} drafted tokens",
        "verify_us": ms_v * 1e3, "verify_gbs": (sbytes + io + wd.B * K * wd.H * 128 * 4) / ms_v / 1e6,
        "commit_us": ms_c * 1e3, "commit_gbs": (2 * sbytes + io) / ms_c / 1e6, "steps": 50}
    del xd, dd, st, vo

    w = gen.WORKLOADS["varlen_64k"]
    x = gen.workload_inputs(w, device=dev)
    cu = gen.cu_seqlens_of(w.seqlens).to(dev)
    a = [x[k][0] for k in ("q", "k", "v", "log_alpha", "beta")]
    o = torch.empty((w.T, w.H, w.dv), dtype=torch.float32, device=dev)
    f = torch.empty((len(w.seqlens), w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    ms = reduce_max(time_call(lambda: binding.kda_varlen_fwd(
        *a, cu, max(w.seqlens), None, out=o, final_state=f), 10, 3, stream), ws)
    res["varlen_64k"] = {"workload": f"{len(w.seqlens)} packed sequences {list(w.seqlens)}, "
                                     f"H={w.H} d={w.dk}",
                         "ms": ms, "Mtok_s": ws * w.T / ms / 1e3, "steps": 10}
    del x, a, o, f
    torch.cuda.empty_cache()
    fixed("long_1m", 3)
    res["long_1m"]["schedule"] = (f"kda_chunk_fwd chooses the segment scan for this shape "
                                  f"({binding.kda_chunk_fwd_launches(1, 1 << 20, 16)} launches)")
    # the same problem with the scan turned off (one segment)
    w = gen.WORKLOADS["long_1m"]
    x = gen.workload_inputs(w, device=dev)
    a = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.float32, device=dev)
    f = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    ms = reduce_max(time_call(lambda: binding.kda_chunk_fwd_segments(
        *a, None, n_segments=1, out=o, final_state=f), 3, 3, stream), ws)
    res["long_1m_without_scan"] = {"workload": "long_1m through kda_chunk_fwd_segments with "
                                               "n_segments=1 (one serial state pass per head)",
                                   "ms": ms, "Mtok_s": ws * w.B * w.T / ms / 1e3, "steps": 3}
    del x, a, o, f
    torch.cuda.empty_cache()
    return res


def run_profile_case(local):
    """Small, fixed case for ncu captures (a few GB on the device at most):
    two prefills of B=1 T=32768 H=32 (long enough for the overlapped,
    segmented schedule), two of the 8k workload (plain two-stage schedule),
    three decode steps, one prefill of B=1 T=131072 H=4, which takes the
    segment scan, then one backward of B=1 T=2048 H=32."""
    from linear_attention_recurrence_fwd_gb300 import binding
    from linear_attention_recurrence_fwd_gb300 import inputs as gen

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    for name, T in (("prefill_64k", 32768), ("prefill_8k", None)):
        w = gen.WORKLOADS[name]
        x = gen.workload_inputs(w, device=dev, T=T)
        a = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
        out = torch.empty(x["v"].shape, dtype=torch.float32, device=dev)
        fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
        for _ in range(2):
            binding.kda_chunk_fwd(*a, x["initial_state"], out=out, final_state=fin)
        torch.cuda.synchronize()
        del x, a, out, fin
    wd = gen.WORKLOADS["decode"]
    xd = gen.make_inputs(wd.B, 1, wd.H, 128, 128, wd.seed, init_std=wd.init_std, device=dev)
    d = [xd[k][:, 0].contiguous() for k in ("q", "k", "v", "log_alpha", "beta")]
    o = torch.empty((wd.B, wd.H, 128), dtype=torch.float32, device=dev)
    for _ in range(3):
        binding.kda_decode_step(*d, xd["initial_state"], out=o)
    torch.cuda.synchronize()
    del xd, d, o
    x = gen.make_inputs(1, 1 << 17, 4, 128, 128, 3, decay_mean=2.0, device=dev)
    binding.kda_chunk_fwd(*[x[k] for k in ("q", "k", "v", "log_alpha", "beta")], None)
    torch.cuda.synchronize()
    del x
    x = gen.make_inputs(1, 2048, 32, 128, 128, 4, init_std=0.02, device=dev)
    d_out = torch.randn((1, 2048, 32, 128), dtype=torch.float32, device=dev,
                        generator=torch.Generator(device=dev).manual_seed(4))
    binding.kda_chunk_bwd(*[x[k] for k in ("q", "k", "v", "log_alpha", "beta")], d_out,
                          initial_state=x["initial_state"])
    torch.cuda.synchronize()
    if binding.kda_last_device_status() != 0:
        raise SystemExit("device status error")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-heads", type=int, default=32)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-extra", action="store_true",
                    help="time only the headline prefill and the decode step")
    ap.add_argument("--case", choices=["bench", "ncu"], default="bench",
                    help="ncu: only run the small profiling case (2 prefills at T=32768 "
                         "and 2 at T=8192, H=32, then 3 decode steps) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.case == "ncu":
        run_profile_case(local)
        return

    from linear_attention_recurrence_fwd_gb300 import binding
    from linear_attention_recurrence_fwd_gb300 import build as kbuild
    from linear_attention_recurrence_fwd_gb300 import inputs as gen

    kbuild.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    stream = torch.cuda.current_stream()

    # ---------------- prefill, T = 65536, H = 32: inputs resident in HBM
    w = gen.WORKLOADS["prefill_64k"]
    x = gen.workload_inputs(w, device=dev)
    args_in = [x[k] for k in ("q", "k", "v", "log_alpha", "beta")]
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.float32, device=dev)
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)

    def step():
        binding.kda_chunk_fwd(*args_in, x["initial_state"], out=out, final_state=fin)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms_local = e0.elapsed_time(e1) / args.steps
    status = binding.kda_last_device_status()
    if status != 0:
        raise SystemExit(f"device status {status}: {binding.kda_status_string(status)}")

    # ---------------- decode: 256 x 32 heads, 1000 chained in-place steps
    wd = gen.WORKLOADS["decode"]
    pool = 64
    xd = gen.make_inputs(wd.B, pool, wd.H, 128, 128, wd.seed, init_std=wd.init_std, device=dev,
                         n_states=wd.B)
    dsets = [[xd[k][:, s].contiguous() for k in ("q", "k", "v", "log_alpha", "beta")]
             for s in range(pool)]
    dstate = xd["initial_state"]
    dout = torch.empty((wd.B, wd.H, 128), dtype=torch.float32, device=dev)
    for s in range(3):
        binding.kda_decode_step(*dsets[s % pool], dstate, out=dout)
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for s in range(args.decode_steps):
        binding.kda_decode_step(*dsets[s % pool], dstate, out=dout)
    d1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    dec_us_local = d0.elapsed_time(d1) * 1e3 / args.decode_steps

    # ---------------- end to end: pinned host inputs -> call -> host output,
    # through the host-buffer entry point (the library copies each round's
    # rows in and its outputs back while other rounds compute)
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in x.items()}
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hfin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    hws = binding.kda_chunk_fwd_host_workspace(w.B, w.T, w.H, w.dk, w.dv, hout.dtype, dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = hout.numel() * hout.element_size() + hfin.numel() * 4

    def e2e_step():
        binding.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                   host["beta"], host["initial_state"], out=hout,
                                   final_state=hfin, workspace=hws)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    g1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms_local = g0.elapsed_time(g1) / args.e2e_steps
    del hws, host

    ms_max = reduce_max(ms_local, ws)
    extra = None
    if not args.skip_extra:
        del out, fin
        extra = extra_workloads(args, ws, dev, stream, x, ms_max)

    launches_per_call = binding.kda_chunk_fwd_launches(w.B, w.T, w.H)
    ms = reduce_max(ms_local, ws)
    dec_us = reduce_max(dec_us_local, ws)
    e2e_ms = reduce_max(e2e_ms_local, ws)
    tokens = w.B * w.T
    value = ws * tokens / (ms * 1e-3) / 1e6
    e2e_value = ws * tokens / (e2e_ms * 1e-3) / 1e6

    if rank != 0:
        return
    alg_bytes = prefill_bytes(tokens, w.H, w.dk, 2, w.B)  # 1282 B per token-head + states
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    f32_bytes = prefill_bytes(tokens, w.H, w.dk, 4, w.B)  # what this run's fp32 output costs
    flops = tokens * w.H * FLOP_PER_TOKEN_HEAD
    tflops = flops / (ms * 1e-3) / 1e12
    dec_bytes = wd.B * wd.H * (2 * 128 * 128 * 4 + 4 * 128 * 2 + 2 + 128 * 4)
    dec_gbs = dec_bytes / (dec_us * 1e-6) / 1e9

    cpu = None
    if not args.skip_cpu:
        sec, cores = oracle_sample(x, args.cpu_heads)
        cpu = {"value": tokens * args.cpu_heads / w.H / sec / 1e6, "unit": "Mtok/s",
               "cores": cores, "kind": "oracle",
               "sample": f"{args.cpu_heads} of {w.H} heads, all {w.T} tokens (fp64, {sec:.1f} s)"}

    line = {
        "metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_64k: B=1 T=65536 H=32 d=128, fp32 out, fp32 state",
                   "B": w.B, "T": w.T, "H": w.H, "d": w.dk, "chunk": 64,
                   "l2": f"inputs larger than L2 ({alg_bytes / 1e9:.2f} GB per step)",
                   "parallelism": f"replicas x{ws}"},
        "tensor": {"tflops": tflops, "frac_burst": tflops / pk["bf16"],
                   "frac_sustained": tflops / pk["bf16_sus"], "peak_src": pk["src"],
                   "flop_per_token_head": FLOP_PER_TOKEN_HEAD},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": achieved / pk["hbm"], "traffic": recorded_traffic(),
                     "alg_bytes_per_launch": alg_bytes,
                     "alg_bytes_note": "1282 B per token-head (q, k, v, log_alpha, beta, "
                                       "bf16 output) + fp32 state in and out",
                     "fp32_output": {"alg_bytes_per_launch": f32_bytes,
                                     "achieved": f32_bytes / (ms * 1e-3) / 1e9,
                                     "frac": f32_bytes / (ms * 1e-3) / 1e9 / pk["hbm"]},
                     "peak_src": pk["src"]},
        "decode": {"us_per_step": dec_us, "state_gbs": dec_gbs, "hbm_frac": dec_gbs / pk["hbm"],
                   "steps": args.decode_steps, "workload": "256 seq x 32 heads x d128, fp32 out"},
        "e2e": {"value": e2e_value, "unit": "Mtok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_call,
        "gpu_launches_note": f"{launches_per_call} per prefill call (the fused launch: state "
                             f"chains and intra-chunk stage in one cooperative grid)"
                             if launches_per_call == 1 else
                             f"{launches_per_call} per prefill call (intra-chunk stage and state "
                             f"pass, per round of the overlapped schedule)",
        "workloads": extra,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
