"""Benchmark: the whole verification + OPD hot path on one batch per step.

Workload (default "mix"): N = 256 requests, L_i ~ U{2,4,8,16} packed by CSR
offsets, V = 151936, bf16 logits (log-Zipf target + Gaussian draft noise).
One step = spec_verify at T = 0 and 0.6, and spec_verify_opd at T = 1 --
verification plus the OPD loss (T = 1, c = 1, lambda = 0.1, forward +
gradient) on the same batch in one pass -- then the adaptive length head:
its label from this round's accepted lengths and its forward pass for the
next round's verified lengths (k = 16, drafter hidden H = 4096, H' = 256,
synthetic hidden states and random weights).  Every step of the path, three
verifications and one loss per step.  The separate T = 1 spec_verify and
opd_loss calls are timed beside it for comparison.

Metric: verified draft positions per second (3 x sum_i L_i per step) for the
whole job; the achieved HBM bandwidth of the dominant kernel is reported in
"roofline" against the measured copy bandwidth.  Inputs (1.2 GB + 1.2 GB of
gradient output per step) are far larger than L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

--impl reference times the CPU oracle (fp64, requests over one thread per core) on a bounded
sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "positions/s"
TEMPS = (0.0, 0.6, 1.0)
OPD = dict(temperature=1.0, clip_c=1.0, lambda_ce=0.1)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.txt")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", choices=["mix"], default="mix")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", choices=["verify_T0", "verify_T0.6", "verify_T1+opd", "length_head"], default=None,
                   help="run warmup + steps iterations of this one call of the step and exit (a small case for "
                        "profilers: no timing, no end-to-end buffers)")
    return p.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_batch(rank: int, **overrides):
    """This rank's batch.  Weak scaling: every rank verifies its own batch of
    the same configuration (independent requests, its own data seed)."""
    import synth
    return synth.config(5, seed=1005 + 7919 * rank, **overrides)


def head_inputs(N: int, rank: int):
    """This rank's length-head inputs (drafter hidden states, random weights)."""
    import synth
    return synth.length_head_inputs(N, HEAD["k"], HEAD["H"], HEAD["Hp"], 2000 + rank)


def reduce_over_ranks(ws: int, dev, elapsed_ms: float, units: float):
    """Job-level timing: the slowest rank's timed region (max) and the units
    all ranks processed (sum).  The only collectives of the run; none is on
    the data path."""
    if ws == 1:
        return float(elapsed_ms), float(units)
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def _src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "serving_vocab_wide_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


KERNEL_SOURCES = {
    "verify_stats": ["verify.cu", "svw_device.cuh", "svw_internal.h"],
    "opd_fast_kernel": ["opd.cu", "opd_common.cuh", "svw_device.cuh", "svw_internal.h"],
}
CALL_KERNELS = {
    "spec_verify": "verify_stats + verify_finalize (accept tests and, at T > 0, the inverse-CDF draw)",
    "opd_loss": "opd_fast_kernel + opd_fix_parts + opd_fix_grad",
    "spec_verify_opd": "opd_fast_kernel (draft rows + bonus rows) + fused_finalize (accept tests, draw) + opd_fix_parts + opd_fix_grad",
    "length_head": "length_head_label + length_head_mma (tcgen05 projection, four K quarters summed in the cluster, bias, SiLU, w2 dot per position) + length_head_final (mean, b2, sigmoid, clamp)",
}
CALLS = ["verify_T0", "verify_T0.6", "verify_T1+opd", "length_head"]
# top-k / top-p settings of the filtered-verification measurement: (T, top_k, top_p)
FILTERS = [(1.0, 50, 0.9), (0.6, 20, 0.95)]
HEAD = dict(k=16, H=4096, Hp=256)
WORKLOAD = ("mix: N=256 ragged L_i~U{2,4,8,16}, V=151936, bf16 log-Zipf logits; verify at T=0 and 0.6, "
            "verify at T=1 fused with OPD fwd/bwd (T=1,c=1,lambda=0.1); length head label + forward "
            "(k=16, H=4096, H'=256)")
CALL_API = {"verify_T0": "spec_verify", "verify_T0.6": "spec_verify", "verify_T1+opd": "spec_verify_opd",
            "length_head": "length_head"}


def _profile_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (same hash) and workload."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    want = _src_hash(KERNEL_SOURCES[kernel])
    for line in open(PROFILE_TRAFFIC, encoding="utf-8"):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") == kernel and f.get("workload") == workload and f.get("src") == want:
            try:
                return float(f["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        time.sleep(0.15)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not getattr(self, "out", ""):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the other workload configurations: one measurement each (their parity is
# tested in tests/); the headline stays on the mix workload
# ---------------------------------------------------------------------------
CONFIG_DESC = {
    1: "tiny: N=4, L=16 (+bonus), V=1024, fp32 logits, T=1 (0.54 MB: L2-resident, latency only)",
    2: "fixed: N=32, L=16 (+bonus), V=151936, bf16, T=1",
    3: "ragged: N=128, L_i~U{2,4,8,16} packed by CSR, V=151936, bf16, T=1",
    4: "opd: 64 requests x 16 draft rows paired 1:1, V=151936, bf16 in, fp32 dlogits, T=1, c=1, lambda=0.1",
}


def _dev_logits(torch, a, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def _time_calls(torch, stream, fn, K):
    """Average time of K back-to-back calls (CUDA events on the launch stream)."""
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return 1000.0 * e0.elapsed_time(e1) / K


def _time_kernel(torch, svw, kernel, fn, K):
    """Average duration of one named kernel inside the call (its own events)."""
    us = []
    for _ in range(K):
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        svw.time_next_launch(kernel, k0, k1)
        fn()
        torch.cuda.synchronize()
        us.append(1000.0 * k0.elapsed_time(k1))
    return float(np.mean(us))


def bench_configs(svw, torch, dev, stream, rank, peak, K=30):
    """spec_verify on workloads 1-3 and opd_loss on workload 4, each with its
    algorithmic bytes (both logit tensors read once; the loss also writes its
    fp32 gradient once), GB/s and fraction of the measured copy bandwidth, for
    the call and for its main kernel."""
    import synth
    out = {}
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    for cfg in (1, 2, 3, 4):
        b = synth.config(cfg, seed=1000 + cfg + 7919 * rank)
        N, R, V = b.N, b.total_rows, b.V
        es = 2 if b.dtype == "bf16" else 4
        code = svw.SVW_BF16 if es == 2 else svw.SVW_F32
        t, d = _dev_logits(torch, b.target, dev), _dev_logits(torch, b.draft, dev)
        cu = torch.from_numpy(b.cu.astype(np.int32)).to(dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if cfg < 4:
            tok = torch.from_numpy(b.tokens[1.0].astype(np.int32)).to(dev)
            acc = torch.empty(N, dtype=torch.int32, device=dev)
            nxt = torch.empty(N, dtype=torch.int32, device=dev)
            ws = torch.empty(svw.verify_workspace_size(N, R, V, code), dtype=torch.uint8, device=dev)

            def fn():
                svw.spec_verify(t, d, cu, tok, 1.0, 0, max_len=16, total_draft_rows=R, accept_len=acc,
                                next_token=nxt, status=st, workspace=ws, stream=stream)
            api, kernel = "spec_verify", "verify_stats"
            alg = (2 * R + N) * V * es
        else:
            loss = torch.empty(R, dtype=torch.float32, device=dev)
            grad = torch.empty((R, V), dtype=torch.float32, device=dev)
            ws = torch.empty(svw.opd_workspace_size(R), dtype=torch.uint8, device=dev)

            def fn():
                svw.opd_loss(t, d, loss=loss, dlogits=grad, status=st, workspace=ws, stream=stream, **OPD)
            api, kernel = "opd_loss", "opd_fast_kernel"
            alg = 2 * R * V * es + R * V * 4
        for _ in range(3):
            fn()
        call_us = _time_calls(torch, stream, fn, K)
        kern_us = _time_kernel(torch, svw, kernel, fn, max(3, K // 2))
        torch.cuda.synchronize()
        rec = {"workload": CONFIG_DESC[cfg], "api": api, "positions": int(R), "call_us": call_us,
               "positions_per_s": R / (call_us * 1e-6), "device_status": int(st.item())}
        if cfg == 1:
            rec["latency_us"] = call_us
        else:
            gbs = alg / (call_us * 1e-6) / 1e9
            kgbs = alg / (kern_us * 1e-6) / 1e9
            rec.update({"algorithmic_bytes": int(alg), "gbs": gbs, "frac_of_peak": gbs / peak,
                        "frac_of_8tbs": gbs / 8000.0, "main_kernel": kernel, "main_kernel_us": kern_us,
                        "main_kernel_gbs": kgbs, "main_kernel_frac_of_peak": kgbs / peak})
        if cfg < 4:
            rec["mean_accept_len"] = float(acc.float().mean().item())
            C = -(-V * es // 36864)  # (row, chunk) items of the stats pass: <= 36 KB chunks
            rec["stats_items"] = int((2 * R + N) * C)
            rec["stats_items_per_sm"] = (2 * R + N) * C / nsm
        out[f"cfg{cfg}"] = rec
        del t, d, ws
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
def launches_per_step():
    """Kernels of this library one step launches: spec_verify = stats +
    finalize, twice; spec_verify_opd = fast pass + finalize + the fix-up's sums
    and gradient grids; length head = label + the tcgen05 projection + the
    per-request finish."""
    return 2 + 2 + 4 + 3


def run_native(args, ws, rank, local):
    import torch
    import serving_vocab_wide_gb300 as svw

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    svw.build()
    svw.lib()
    b = make_batch(rank)
    N, R, V = b.N, b.total_rows, b.V
    rows_t = R + N

    def logits_host(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    h_t = logits_host(b.target)
    h_d = logits_host(b.draft)
    h_cu = torch.from_numpy(b.cu.astype(np.int32)).pin_memory()
    h_tok = {T: torch.from_numpy(b.tokens[T].astype(np.int32)).pin_memory() for T in TEMPS}
    t = h_t.to(dev)
    d = h_d.to(dev)
    cu = h_cu.to(dev)
    tok = {T: h_tok[T].to(dev) for T in TEMPS}
    ws_bytes = svw.verify_workspace_size(N, R, V, svw.SVW_BF16)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    opd_ws = torch.empty(svw.opd_workspace_size(R), dtype=torch.uint8, device=dev)
    fused_ws = torch.empty(svw.verify_opd_workspace_size(N, R, V, svw.SVW_BF16), dtype=torch.uint8, device=dev)
    # adaptive length head: synthetic drafter hidden states and random weights
    hk, hH, hHp = HEAD["k"], HEAD["H"], HEAD["Hp"]
    hin = head_inputs(N, rank)
    h_hid = torch.from_numpy(hin["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hid = h_hid.to(dev)
    w1 = torch.from_numpy(hin["w1"].view(np.int16)).view(torch.bfloat16).to(dev)
    b1 = torch.from_numpy(hin["b1"]).to(dev)
    w2 = torch.from_numpy(hin["w2"]).to(dev)
    head_ws = torch.empty(svw.lib().svw_length_head_workspace_size(N, hk, hHp), dtype=torch.uint8, device=dev)
    a_hat = torch.empty(N, dtype=torch.float32, device=dev)
    k_hat = torch.empty(N, dtype=torch.int32, device=dev)
    a_star = torch.empty(N, dtype=torch.float32, device=dev)
    len_loss = torch.empty(N, dtype=torch.float32, device=dev)
    acc = {T: torch.empty(N, dtype=torch.int32, device=dev) for T in TEMPS}
    nxt = {T: torch.empty(N, dtype=torch.int32, device=dev) for T in TEMPS}
    loss = torch.empty(R, dtype=torch.float32, device=dev)
    grad = torch.empty((R, V), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    calls = CALLS

    # the input set the step reads (the end-to-end loop alternates two)
    cur = [dict(t=t, d=d, cu=cu, tok=tok, hid=hid)]

    def verify(T):
        x = cur[0]
        svw.spec_verify(x["t"], x["d"], x["cu"], x["tok"][T], T, 0, max_len=16, total_draft_rows=R,
                        accept_len=acc[T], next_token=nxt[T], status=status, workspace=wsp, stream=stream)

    def verify_opd():
        x = cur[0]
        svw.spec_verify_opd(x["t"], x["d"], x["cu"], x["tok"][1.0], 1.0, 0, opd_temperature=OPD["temperature"],
                            clip_c=OPD["clip_c"], lambda_ce=OPD["lambda_ce"], max_len=16,
                            total_draft_rows=R, accept_len=acc[1.0], next_token=nxt[1.0], loss=loss,
                            dlogits=grad, status=status, workspace=fused_ws, stream=stream)

    # the main kernel of each call, timed inside the call (svw_time_next_launch)
    call_kernel = {"verify_T0": "verify_stats", "verify_T0.6": "verify_stats", "verify_T1+opd": "opd_fast_kernel",
                   "length_head": "length_head_mma"}

    def head():
        # this round's label (T = 1 accepted lengths against last round's a_hat), then the
        # forward pass that sets the next round's verified lengths
        x = cur[0]
        svw.length_head_label(acc[1.0], x["cu"], a_hat, a_star=a_star, loss=len_loss, stream=stream)
        svw.length_head(x["hid"], w1, b1, w2, hin["b2"], hin["gamma"], a_hat=a_hat, k_hat=k_hat,
                        workspace=head_ws, stream=stream)

    def step(ev=None, kev=None):
        for ci, fn in enumerate((lambda: verify(0.0), lambda: verify(0.6), verify_opd, head)):
            if kev is not None:
                svw.time_next_launch(call_kernel[calls[ci]], kev[2 * ci], kev[2 * ci + 1])
            if ev is not None:
                ev[2 * ci].record(stream)
            fn()
            if ev is not None:
                ev[2 * ci + 1].record(stream)

    if args.only is not None:
        fn = dict(zip(calls, (lambda: verify(0.0), lambda: verify(0.6), verify_opd, head)))[args.only]
        for _ in range(args.warmup + args.steps):
            fn()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"only": args.only, "iterations": args.warmup + args.steps,
                              "device_status": int(status.item())}))
        return

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    # ---- device-timed region: inputs resident in HBM ----
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(calls))] for _ in range(K)]

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for k in range(K):
            step(evs[k])
        e1.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    positions_per_step = 3 * R
    elapsed_ms, job_positions = reduce_over_ranks(ws, dev, e0.elapsed_time(e1), positions_per_step)
    per_call = {c: [] for c in calls}
    for k in range(K):
        for ci, c in enumerate(calls):
            per_call[c].append(evs[k][2 * ci].elapsed_time(evs[k][2 * ci + 1]))
    avg_us = {c: 1000.0 * float(np.mean(v)) for c, v in per_call.items()}
    # ---- each call's main kernel on its own, in a second timed loop (recording
    # events between kernels would hold back the programmatic launches of the
    # first loop) ----
    Kk = max(3, min(K, 50))
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(calls))] for _ in range(Kk)]
    for k in range(Kk):
        step(None, kevs[k])
    torch.cuda.synchronize()
    kern_us = {c: 1000.0 * float(np.mean([kevs[k][2 * ci].elapsed_time(kevs[k][2 * ci + 1]) for k in range(Kk)]))
               for ci, c in enumerate(calls)}

    # algorithmic bytes per call (each logit byte read once; the loss also
    # writes its fp32 gradient once)
    es = 2
    alg = {"verify_T0": rows_t * V * es,
           "verify_T0.6": (rows_t + R) * V * es,
           "verify_T1+opd": (rows_t + R) * V * es + R * V * 4,
           "verify_T1": (rows_t + R) * V * es,
           "opd": 2 * R * V * es + R * V * 4,
           "length_head": N * hk * hH * 2 + hHp * hH * 2 + N * hk * hHp * 4 * 2}
    ms_per_step = elapsed_ms / K
    value = job_positions / (elapsed_ms / K / 1000.0)
    step_bytes = sum(alg[c] for c in calls)
    peak, peak_kind = _peaks()
    # the dominant kernel: the longest main kernel of a call, timed on the
    # launch stream inside the call; its algorithmic bytes
    kalg = {"verify_T0": alg["verify_T0"], "verify_T0.6": alg["verify_T0.6"],
            "verify_T1+opd": 2 * R * V * es + R * V * 4 + N * V * es,
            "length_head": N * hk * hH * 2 + hHp * hH * 2 + N * hk * hHp * 4}
    head_flops = 2.0 * N * hk * hH * hHp
    dom = max((c for c in calls if c != "length_head"), key=lambda c: kern_us[c])
    dom_kernel = call_kernel[dom]
    achieved = kalg[dom] / (kern_us[dom] * 1e-6) / 1e9
    traffic = _profile_traffic(dom_kernel, f"mix:{dom}")

    # ---- for comparison: the T = 1 verification and the loss as two calls ----
    Ks = max(3, min(K, 30))
    sep = {}
    for name, fn in (("verify_T1", lambda: verify(1.0)),
                     ("opd", lambda: svw.opd_loss(t, d, cu_draft=cu, has_bonus=True, loss=loss, dlogits=grad,
                                                  status=status, workspace=opd_ws, stream=stream, **OPD))):
        fn()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(Ks):
            fn()
        s1.record(stream)
        torch.cuda.synchronize()
        us = 1000.0 * s0.elapsed_time(s1) / Ks
        sep[name] = {"avg_us": us, "gbs": alg[name] / (us * 1e-6) / 1e9}
    sep["sum_us"] = sep["verify_T1"]["avg_us"] + sep["opd"]["avg_us"]

    # ---- early-exit verification of the same batch: the same accepted lengths
    # and tokens from the rows up to each request's first rejection ----
    early_ws = torch.empty(svw.verify_early_workspace_size(N, R, V, svw.SVW_BF16), dtype=torch.uint8, device=dev)
    nbytes = torch.zeros(1, dtype=torch.int64, device=dev)
    acc_e = torch.empty(N, dtype=torch.int32, device=dev)
    nxt_e = torch.empty(N, dtype=torch.int32, device=dev)
    full_us = {0.0: avg_us["verify_T0"], 0.6: avg_us["verify_T0.6"], 1.0: sep["verify_T1"]["avg_us"]}
    early = {}
    for T in TEMPS:
        def fn():
            svw.spec_verify_early(t, d, cu, tok[T], T, 0, max_len=16, total_draft_rows=R, accept_len=acc_e,
                                  next_token=nxt_e, status=status, bytes_read=nbytes, workspace=early_ws,
                                  stream=stream)
        fn()
        torch.cuda.synchronize()
        differ = int(((acc_e != acc[T]) | (nxt_e != nxt[T])).sum().item())
        read = int(nbytes.item())
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(Ks):
            fn()
        s1.record(stream)
        torch.cuda.synchronize()
        us = 1000.0 * s0.elapsed_time(s1) / Ks
        kus = []
        for _ in range(Ks):
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            svw.time_next_launch("verify_early_cluster", k0, k1)
            fn()
            torch.cuda.synchronize()
            kus.append(1000.0 * k0.elapsed_time(k1))
        kus = float(np.mean(kus))
        full_bytes = (rows_t if T == 0.0 else rows_t + R) * V * 2
        early[f"T{T:g}"] = {"avg_us": us, "effective_positions_per_s": R / (us * 1e-6),
                            "full_read_call_us": full_us[T], "speedup_vs_full_read": full_us[T] / us,
                            "bytes_read": read, "read_frac": read / full_bytes,
                            "kernel": "verify_early_cluster", "kernel_us": kus,
                            "kernel_gbs": read / (kus * 1e-6) / 1e9,
                            "requests_differing_from_spec_verify": differ}

    # ---- top-k / top-p filtered verification of the same batch (draft tokens
    # redrawn from the filtered draft distribution) ----
    filt_ws = torch.empty(svw.verify_filtered_workspace_size(N, R, V, svw.SVW_BF16), dtype=torch.uint8,
                          device=dev)
    filtered = {}
    for T, kf, pf in FILTERS:
        import synth
        ftok = torch.from_numpy(synth.sample_tokens_filtered(b.draft, T, kf, pf, 4000 + rank)).to(dev)

        def fn():
            svw.spec_verify_filtered(t, d, cu, ftok, T, kf, pf, 0, max_len=16, total_draft_rows=R,
                                     accept_len=acc_e, next_token=nxt_e, status=status, workspace=filt_ws,
                                     stream=stream)
        fn()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(Ks):
            fn()
        s1.record(stream)
        torch.cuda.synchronize()
        us = 1000.0 * s0.elapsed_time(s1) / Ks
        kus = []
        for _ in range(Ks):
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            svw.time_next_launch("filter_rows", k0, k1)
            fn()
            torch.cuda.synchronize()
            kus.append(1000.0 * k0.elapsed_time(k1))
        kus = float(np.mean(kus))
        rows_bytes = (rows_t + R) * V * 2
        filtered[f"T{T:g}_k{kf}_p{pf:g}"] = {
            "avg_us": us, "positions_per_s": R / (us * 1e-6), "kernel": "filter_rows", "kernel_us": kus,
            "kernel_gbs": rows_bytes / (kus * 1e-6) / 1e9, "algorithmic_bytes": rows_bytes,
            "mean_accept_len": float(acc_e.float().mean().item())}

    # ---- end to end through the public API with host buffers ----
    Ke = args.e2e_steps if args.e2e_steps is not None else max(3, min(K, 60))
    h_acc = {T: torch.empty(N, dtype=torch.int32).pin_memory() for T in TEMPS}
    h_nxt = {T: torch.empty(N, dtype=torch.int32).pin_memory() for T in TEMPS}
    h_loss = torch.empty(R, dtype=torch.float32).pin_memory()
    h_khat = torch.empty(N, dtype=torch.int32).pin_memory()

    # double-buffered inputs: step k+1's host-to-device copies run on a copy
    # stream while step k's kernels run; every step's copies and result reads
    # are inside the timed region
    sets = [cur[0], dict(t=torch.empty_like(t), d=torch.empty_like(d), cu=torch.empty_like(cu),
                         tok={T: torch.empty_like(tok[T]) for T in TEMPS}, hid=torch.empty_like(hid))]
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    free = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d_into(s):
        x = sets[s]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[s])  # the set's previous step is done reading it
            x["t"].copy_(h_t, non_blocking=True)
            x["d"].copy_(h_d, non_blocking=True)
            x["cu"].copy_(h_cu, non_blocking=True)
            for T in TEMPS:
                x["tok"][T].copy_(h_tok[T], non_blocking=True)
            x["hid"].copy_(h_hid, non_blocking=True)
            ready[s].record(copy_stream)

    def run_on(s):
        stream.wait_event(ready[s])
        cur[0] = sets[s]
        step()
        free[s].record(stream)
        for T in TEMPS:
            h_acc[T].copy_(acc[T], non_blocking=True)
            h_nxt[T].copy_(nxt[T], non_blocking=True)
        h_loss.copy_(loss, non_blocking=True)
        h_khat.copy_(k_hat, non_blocking=True)

    def e2e_run(n):
        copy_stream.wait_stream(stream)
        h2d_into(0)
        for k in range(n):
            if k + 1 < n:
                h2d_into((k + 1) % 2)
            run_on(k % 2)

    e2e_run(2)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_run(Ke)
    f1.record(stream)
    torch.cuda.synchronize()
    cur[0] = sets[0]
    e2e_ms, _ = reduce_over_ranks(ws, dev, f0.elapsed_time(f1), positions_per_step)
    h2d = ((h_t.numel() + h_d.numel()) * 2 + h_cu.numel() * 4 + sum(v.numel() * 4 for v in h_tok.values())
           + h_hid.numel() * 2)
    d2h = 2 * 3 * N * 4 + R * 4 + N * 4
    e2e = {"value": job_positions / (e2e_ms / Ke / 1000.0), "unit": UNIT,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": Ke,
           "pipelining": "double-buffered inputs: step k+1's host-to-device copies overlap step k's kernels"}

    status_v = int(status.item())
    gpu_acc = {T: acc[T].cpu().numpy() for T in TEMPS}
    gpu_nxt = {T: nxt[T].cpu().numpy() for T in TEMPS}

    # ---- the other workload configurations (parity cases of their own; one
    # number each, not part of the step) ----
    configs = bench_configs(svw, torch, dev, stream, rank, peak)

    cpu = None
    cpu_all = None
    ties = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(b, hin)
        cpu_all = cpu_baseline_all_cores(b, hin)
        ties = near_ties(b, gpu_acc, gpu_nxt)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "N": N, "total_draft_rows": R, "V": V, "logits": "bf16",
                   "per_rank_batch": True, "parallelism": f"replicas x{ws}",
                   "l2": "inputs 1.25 GB per step > 129 MB L2; no flush"},
        "roofline": {"bound": "hbm", "kernel": f"{dom_kernel} (in {CALL_API[dom]}, {dom})",
                     "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": kalg[dom], "avg_launch_us": kern_us[dom]},
        "length_head_mma": {"tflops": head_flops / (kern_us["length_head"] * 1e-6) / 1e12,
                             "avg_us": kern_us["length_head"], "unit": "TFLOP/s",
                             "peak_bf16": _peak_tflops(), "frac": head_flops / (kern_us["length_head"] * 1e-6)
                             / 1e12 / _peak_tflops()},
        "calls": {c: {"api": CALL_API[c], "kernels": CALL_KERNELS[CALL_API[c]], "avg_us": avg_us[c],
                      "gbs": alg[c] / (avg_us[c] * 1e-6) / 1e9,
                      "frac_of_peak": alg[c] / (avg_us[c] * 1e-6) / 1e9 / peak,
                      "main_kernel": call_kernel[c], "main_kernel_us": kern_us[c],
                      "main_kernel_gbs": kalg[c] / (kern_us[c] * 1e-6) / 1e9}
                  for c in calls},
        "separate_calls": sep,
        "early_exit": early,
        "filtered": filtered,
        "step_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "e2e": e2e,
        "gpu_launches": K * launches_per_step(),
        "clocks": clk.summary(),
        "device_status": status_v,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "near_ties": ties,
        "configs": configs,
    }
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def _oracle_sample(b, n_req):
    sub = b.subset(range(n_req))
    return sub, np.arange(n_req, dtype=np.int32)


def oracle_step(sub, ids, head):
    """One step of the oracle on requests `ids`: the three verifications, the
    OPD loss and gradient, and the length head's label and forward pass --
    the same work as one native step."""
    import oracle
    acc = None
    for T in TEMPS:
        r = oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[T], T, 0, max_len=16, req_ids=ids)
        if T == 1.0:
            acc = r["accept_len"]
    oracle.opd_loss(sub.target, sub.draft, cu_draft=sub.cu, has_bonus=True, **OPD)
    h = oracle.length_head(head["hidden"][ids], head["w1"], head["b1"], head["w2"], head["b2"], head["gamma"])
    oracle.length_label(acc, sub.cu, h["a_hat"])


def cpu_baseline(b, head, n_req=40):
    """Oracle timed on a bounded sample: the first n_req requests of the batch,
    one full step (three verifications, the OPD loss + gradient, the length
    head)."""
    import oracle
    oracle.build()
    sub, ids = _oracle_sample(b, n_req)
    t0 = time.perf_counter()
    oracle_step(sub, ids, head)
    dt = time.perf_counter() - t0
    return {"value": 3 * sub.total_rows / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {n_req} requests ({sub.total_rows} positions) of the mix batch, "
                      f"one step: verify T=0,0.6,1 + OPD fwd/bwd + length head; {dt:.1f} s"}


def _host_cores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _oracle_groups(b, n_req, nt):
    """n_req requests of the batch split into nt contiguous groups (one per
    thread); each group is a batch of its own with its original request ids."""
    bounds = np.linspace(0, n_req, nt + 1).astype(int)
    groups = []
    for g in range(nt):
        ids = np.arange(bounds[g], bounds[g + 1], dtype=np.int32)
        if ids.size:
            groups.append((b.subset(ids), ids))
    return groups


def oracle_step_threads(groups, pool, head):
    """One step of the unchanged oracle, its requests spread over threads (the
    requests are independent; the C calls release the GIL)."""
    list(pool.map(lambda g: oracle_step(g[0], g[1], head), groups))


def cpu_baseline_all_cores(b, head):
    """The oracle on every request of the batch, one thread per host core."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    oracle._load()
    nt = _host_cores()
    groups = _oracle_groups(b, b.N, nt)
    rows = sum(g[0].total_rows for g in groups)
    with ThreadPoolExecutor(max_workers=nt) as pool:
        t0 = time.perf_counter()
        oracle_step_threads(groups, pool, head)
        dt = time.perf_counter() - t0
    return {"value": 3 * rows / dt, "unit": UNIT, "cores": nt, "kind": "oracle",
            "sample": f"all {b.N} requests ({rows} positions) of the mix batch, one step: verify T=0,0.6,1 "
                      f"+ OPD fwd/bwd + length head, requests split over {nt} threads; {dt:.1f} s"}


NEAR_BAND = 1e-5


def near_ties(b, acc, nxt):
    """The oracle's near-tie flags on the whole batch at each temperature of
    the step, against the GPU's results (one oracle pass per temperature on
    all host cores, outside any timed region): requests flagged near an
    accept threshold / a CDF boundary (band 1e-5), how many of them the GPU
    decided differently, and whether each such difference is within the band
    (the oracle's distance from its draw point to the GPU token's CDF
    interval).  Unflagged differences would be parity failures."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    nt = _host_cores()
    groups = _oracle_groups(b, b.N, 4 * nt)
    out = {}
    for T in TEMPS:
        def work(g):
            sub, ids = g
            return ids, oracle.spec_verify(sub.target, sub.draft, sub.cu, sub.tokens[T], T, 0, max_len=16,
                                           req_ids=ids, alt_next=nxt[T][ids])
        with ThreadPoolExecutor(max_workers=nt) as pool:
            res = list(pool.map(work, groups))
        fl = np.zeros(b.N, np.int32)
        ra = np.zeros(b.N, np.int32)
        rn = np.zeros(b.N, np.int32)
        dist = np.zeros(b.N)
        for ids, r in res:
            fl[ids], ra[ids], rn[ids], dist[ids] = r["flags"], r["accept_len"], r["next_token"], r["alt_dist"]
        near = (fl & (oracle.FLAG_NEAR_ACCEPT | oracle.FLAG_NEAR_CDF | oracle.FLAG_DEGENERATE)) != 0
        diff = (acc[T] != ra) | (nxt[T] != rn)
        tok_diff = diff & (acc[T] == ra)
        out[f"T{T:g}"] = {
            "requests": int(b.N), "band": NEAR_BAND,
            "flagged_near_accept": int(((fl & oracle.FLAG_NEAR_ACCEPT) != 0).sum()),
            "flagged_near_cdf": int(((fl & oracle.FLAG_NEAR_CDF) != 0).sum()),
            "flagged_and_differing": int((diff & near).sum()),
            "unflagged_differing": int((diff & ~near).sum()),
            "differing_tokens_within_band": bool(np.all(dist[tok_diff] <= NEAR_BAND)),
        }
    return out


def run_reference(args, ws, rank):
    """The oracle as it stands, timed on the host cores: each step is a bounded
    sample of the mix batch, its requests split over one thread per core."""
    if rank != 0:
        return
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    oracle._load()
    b = make_batch(0)
    head = head_inputs(b.N, 0)
    nt = _host_cores()
    # size each step's sample so that warmup + steps finish in about 90 s
    probe, pids = _oracle_sample(b, 1)
    t0 = time.perf_counter()
    oracle_step(probe, pids, head)
    per_req = max(1e-3, time.perf_counter() - t0)
    n_req = int(max(1, min(b.N, 90.0 * nt / (per_req * max(1, args.steps + args.warmup)))))
    groups = _oracle_groups(b, n_req, nt)
    rows = sum(g[0].total_rows for g in groups)
    with ThreadPoolExecutor(max_workers=nt) as pool:
        for _ in range(args.warmup):
            oracle_step_threads(groups, pool, head)
        K = args.steps
        t0 = time.perf_counter()
        for _ in range(K):
            oracle_step_threads(groups, pool, head)
        dt = (time.perf_counter() - t0) / K
    value = 3 * rows / dt
    sample = (f"first {n_req} requests ({rows} positions) of the mix batch per step (verify T=0,0.6,1 + "
              f"OPD fwd/bwd + length head), fp64 oracle, requests split over {nt} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": dt * 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_native(args, ws, rank, local)


if __name__ == "__main__":
    main()
